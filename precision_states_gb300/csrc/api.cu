// api.cu -- the device-facing part of the C ABI: plan creation (validation,
// chunk table, one workspace allocation, upload), the gradient norm, the
// fused steps, and the standalone codecs.  Every argument is checked on the
// host before anything is launched; failures return a status and launch
// nothing.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "internal.h"

using namespace psopt;

// Each wait of the staged step kernel gives up after this long unless the
// plan sets another limit (opt_plan_set_wait_limit).
constexpr uint64_t kDefaultWaitNs = 2000000000ull;      // 2 s
constexpr uint64_t kMaxWaitNs = 10000000000ull;         // 10 s

struct opt_plan {
  int device = 0;
  int sm_count = 0;
  int32_t n = 0;
  int64_t total_numel = 0;
  int64_t n_chunks = 0;
  int64_t bucket_begin[3] = {0, 0, 0};       // norm chunks per gradient-dtype bucket
  int64_t n_tiles = 0;
  int64_t tile_begin[3] = {0, 0, 0};         // step tiles per bucket
  int32_t m_dtype = OPT_F32, v_dtype = OPT_F32;
  int combo = SC_F32;
  bool has_m2 = false;
  // per gradient-dtype bucket: the whole bucket as kernel parameters, when
  // it is short enough for the short-list step (small_ok)
  SmallList small[2];
  bool small_ok[2] = {false, false};
  std::vector<void*> grad_dev;          // per tensor, for opt_grads_upload
  std::vector<int64_t> grad_bytes;
  // one device allocation: tensors | norm chunks | tiles | slots | result | counter | flags |
  // norm completion counter | step counter | step scalars
  void* d_mem = nullptr;
  int64_t d_bytes = 0;
  TensorDesc* d_tensors = nullptr;
  NormChunk* d_chunks = nullptr;           // the norm's chunks, addresses resolved
  opt_chunk* d_tiles = nullptr;
  NormSlot* d_slots = nullptr;
  opt_norm_result* d_result = nullptr;
  unsigned long long* d_unchanged = nullptr;
  int* d_err = nullptr;                    // kernel error flags (opt_plan_status)
  uint64_t wait_ns = kDefaultWaitNs;       // limit of each wait of the staged step
  unsigned int* d_done = nullptr;          // the norm's completion counter
  int64_t* d_step = nullptr;               // device step counter (last step taken)
  opt_step_scalars* d_sc = nullptr;        // its step's scalars
  unsigned long long* d_dyn = nullptr;     // the warp-dynamic step's counters (0 between launches)
  // update-norm clipping (LAMB) workspace, allocated on first use
  std::vector<int64_t> tile_first, tile_count;   // per tensor, in the tile table
  void* d_lamb = nullptr;
  psopt::LambWork lamb{};
};

namespace psopt {
int state_combo(int32_t m_dtype, int32_t v_dtype) {
  if (m_dtype == OPT_F32 && v_dtype == OPT_F32) return SC_F32;
  if (m_dtype == OPT_BF16 && v_dtype == OPT_BF16) return SC_BF16_BF16;
  if (m_dtype == OPT_BF16 && v_dtype == OPT_E4M3) return SC_BF16_E4M3;
  if (m_dtype == OPT_BF16 && v_dtype == OPT_E2M2) return SC_BF16_E2M2;
  return -1;
}
}  // namespace psopt

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int64_t state_bytes(int32_t dtype, int64_t n) {
  switch (dtype) {
    case OPT_F32: return 4 * n;
    case OPT_BF16: return 2 * n;
    case OPT_E4M3: return n;
    case OPT_E2M2: return (n + 1) / 2;
  }
  return -1;
}

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return OPT_OK;
  if (e == cudaErrorMemoryAllocation) return OPT_ENOMEM;
  return OPT_ECUDA;
}

// Make the plan's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// A usable v scale: a positive power of two whose reciprocal is also a
// normal float, so both scalings are exact.
bool valid_scale(float s) {
  if (!(s > 0.0f) || !std::isfinite(s)) return false;
  int e = 0;
  return std::frexp(s, &e) == 0.5f && e >= -100 && e <= 100;
}

int validate_list(const opt_tensor_list* L) {
  if (L == nullptr || L->n < 0) return OPT_EINVAL;
  if (L->n > 0 && (L->numel == nullptr || L->param == nullptr || L->grad == nullptr ||
                   L->m == nullptr || L->v == nullptr || L->grad_dtype == nullptr))
    return OPT_EINVAL;
  if (L->param_dtype != OPT_F32) return OPT_EUNSUPPORTED;
  if (state_combo(L->m_dtype, L->v_dtype) < 0) return OPT_EUNSUPPORTED;
  for (int32_t i = 0; i < L->n; ++i) {
    if (L->numel[i] < 0) return OPT_EINVAL;
    if (L->v_scale != nullptr && !valid_scale(L->v_scale[i])) return OPT_EINVAL;
    if (L->v_scale != nullptr && L->v_dtype == OPT_F32 && L->v_scale[i] != 1.0f) return OPT_EINVAL;
    if (L->grad_dtype[i] != OPT_F32 && L->grad_dtype[i] != OPT_BF16) return OPT_EUNSUPPORTED;
    if (L->numel[i] == 0) continue;
    const void* ptrs[5] = {L->param[i], L->grad[i], L->m[i], L->v[i],
                           L->m2 ? L->m2[i] : nullptr};
    for (int k = 0; k < 4; ++k)
      if (ptrs[k] == nullptr) return OPT_EINVAL;
    for (int k = 0; k < 5; ++k)
      if (ptrs[k] != nullptr && !aligned16(ptrs[k])) return OPT_EALIGN;
  }
  return OPT_OK;
}

}  // namespace

extern "C" {

int opt_plan_create(const opt_tensor_list* L, opt_plan** out) {
  if (out == nullptr) return OPT_EINVAL;
  *out = nullptr;
  int st = validate_list(L);
  if (st != OPT_OK) return st;

  opt_plan* P = new (std::nothrow) opt_plan();
  if (P == nullptr) return OPT_ENOMEM;
  P->n = L->n;
  P->m_dtype = L->m_dtype;
  P->v_dtype = L->v_dtype;
  P->combo = state_combo(L->m_dtype, L->v_dtype);
  P->has_m2 = L->m2 != nullptr;
  if (P->has_m2)
    for (int32_t i = 0; i < L->n; ++i)
      if (L->numel[i] > 0 && L->m2[i] == nullptr) P->has_m2 = false;

  // chunk table on the host, from sizes only
  int64_t nch = opt_chunk_table(L->n, L->numel, L->grad_dtype, nullptr, 0, P->bucket_begin);
  if (nch < 0) { delete P; return (int)nch; }
  std::vector<opt_chunk> chunks((size_t)nch);
  opt_chunk_table(L->n, L->numel, L->grad_dtype, chunks.data(), nch, P->bucket_begin);
  P->n_chunks = nch;
  const int64_t tile_elems[2] = {kTileElems, kTileElems};
  const int64_t ntl = build_table(L->n, L->numel, L->grad_dtype, tile_elems, nullptr, 0, P->tile_begin);
  std::vector<opt_chunk> tiles((size_t)ntl);
  build_table(L->n, L->numel, L->grad_dtype, tile_elems, tiles.data(), ntl, P->tile_begin);
  P->n_tiles = ntl;
  P->tile_first.assign((size_t)L->n, 0);
  P->tile_count.assign((size_t)L->n, 0);
  for (int64_t k = ntl - 1; k >= 0; --k) {     // a tensor's tiles are contiguous
    P->tile_first[tiles[(size_t)k].tensor] = k;
    P->tile_count[tiles[(size_t)k].tensor] += 1;
  }

  std::vector<TensorDesc> tds((size_t)L->n);
  P->grad_dev.resize((size_t)L->n);
  P->grad_bytes.resize((size_t)L->n);
  for (int32_t i = 0; i < L->n; ++i) {
    TensorDesc& t = tds[(size_t)i];
    t.p = static_cast<float*>(L->param[i]);
    t.g = L->grad[i];
    t.m = L->m[i];
    t.v = L->v[i];
    t.m2 = P->has_m2 ? static_cast<float*>(L->m2[i]) : nullptr;
    t.numel = L->numel[i];
    t.v_scale = L->v_scale ? L->v_scale[i] : 1.0f;
    t.v_inv_scale = 1.0f / t.v_scale;     // exact for a power of two
    // FP32 p, m, v that start on a 32-byte boundary take 32-byte loads in
    // the AdamW step
    auto a32 = [](const void* q) { return ((uintptr_t)q & 31u) == 0; };
    t.a32 = (a32(t.p) ? kA32P : 0u) | (L->m_dtype == OPT_F32 && a32(t.m) ? kA32M : 0u) |
            (L->v_dtype == OPT_F32 && a32(t.v) ? kA32V : 0u);
    t.pad = 0;
    P->total_numel += L->numel[i];
    P->grad_dev[(size_t)i] = const_cast<void*>(L->grad[i]);
    P->grad_bytes[(size_t)i] = state_bytes(L->grad_dtype[i], L->numel[i]);
  }

  // short buckets for the short-list step: at most kSmallMaxTensors
  // non-empty tensors and kSmallMaxTiles tiles, in list order
  for (int b = 0; b < 2; ++b) {
    SmallList& sl = P->small[b];
    std::memset(&sl, 0, sizeof sl);
    int64_t tiles = 0;
    bool ok = true;
    for (int32_t i = 0; i < L->n && ok; ++i) {
      if (L->numel[i] == 0 || (L->grad_dtype[i] == OPT_BF16 ? 1 : 0) != b) continue;
      if (sl.n == kSmallMaxTensors) { ok = false; break; }
      tiles += (L->numel[i] + kTileElems - 1) / kTileElems;
      sl.tensor[sl.n] = (uint32_t)i;
      sl.tile_end[sl.n] = tiles;
      sl.td[sl.n] = tds[(size_t)i];
      sl.n += 1;
    }
    P->small_ok[b] = ok && sl.n > 0 && tiles <= kSmallMaxTiles;
  }

  // the norm's table: each chunk's first gradient element, resolved
  std::vector<NormChunk> nchunks((size_t)nch);
  for (int64_t k = 0; k < nch; ++k) {
    const opt_chunk& c = chunks[(size_t)k];
    const int64_t esize = L->grad_dtype[c.tensor] == OPT_BF16 ? 2 : 4;
    nchunks[(size_t)k].ptr = static_cast<const char*>(L->grad[c.tensor]) + c.start * esize;
    nchunks[(size_t)k].len = c.len;
    nchunks[(size_t)k].pad = 0;
  }

  if (cudaGetDevice(&P->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&P->sm_count, cudaDevAttrMultiProcessorCount, P->device) != cudaSuccess) {
    delete P;
    return OPT_ECUDA;
  }

  const int64_t off_t = 0;
  const int64_t off_c = align_up(off_t + (int64_t)sizeof(TensorDesc) * L->n, 256);
  const int64_t off_l = align_up(off_c + (int64_t)sizeof(NormChunk) * nch, 256);
  const int64_t off_s = align_up(off_l + (int64_t)sizeof(opt_chunk) * ntl, 256);
  const int64_t off_r = align_up(off_s + (int64_t)sizeof(NormSlot) * 2 * OPT_NORM_SLOTS, 256);
  const int64_t off_u = align_up(off_r + (int64_t)sizeof(opt_norm_result), 256);
  const int64_t off_e = off_u + 8;
  const int64_t off_d = off_e + 8;
  const int64_t off_k = align_up(off_d + 8, 16);
  const int64_t off_q = off_k + 16;
  const int64_t off_y = align_up(off_q + (int64_t)sizeof(opt_step_scalars), 16);
  P->d_bytes = align_up(off_y + 16, 256);
  cudaError_t e = cudaMalloc(&P->d_mem, (size_t)P->d_bytes);
  if (e != cudaSuccess) { delete P; return cuda_status(e); }
  char* base = static_cast<char*>(P->d_mem);
  P->d_tensors = reinterpret_cast<TensorDesc*>(base + off_t);
  P->d_chunks = reinterpret_cast<NormChunk*>(base + off_c);
  P->d_tiles = reinterpret_cast<opt_chunk*>(base + off_l);
  P->d_slots = reinterpret_cast<NormSlot*>(base + off_s);
  P->d_result = reinterpret_cast<opt_norm_result*>(base + off_r);
  P->d_unchanged = reinterpret_cast<unsigned long long*>(base + off_u);
  P->d_err = reinterpret_cast<int*>(base + off_e);
  P->d_done = reinterpret_cast<unsigned int*>(base + off_d);
  P->d_step = reinterpret_cast<int64_t*>(base + off_k);
  P->d_sc = reinterpret_cast<opt_step_scalars*>(base + off_q);
  P->d_dyn = reinterpret_cast<unsigned long long*>(base + off_y);

  e = cudaMemset(P->d_mem, 0, (size_t)P->d_bytes);
  if (e == cudaSuccess && L->n > 0)
    e = cudaMemcpy(P->d_tensors, tds.data(), sizeof(TensorDesc) * (size_t)L->n, cudaMemcpyHostToDevice);
  if (e == cudaSuccess && nch > 0)
    e = cudaMemcpy(P->d_chunks, nchunks.data(), sizeof(NormChunk) * (size_t)nch, cudaMemcpyHostToDevice);
  if (e == cudaSuccess && ntl > 0)
    e = cudaMemcpy(P->d_tiles, tiles.data(), sizeof(opt_chunk) * (size_t)ntl, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(P->d_mem);
    delete P;
    return cuda_status(e);
  }
  *out = P;
  return OPT_OK;
}

void opt_plan_destroy(opt_plan* P) {
  if (P == nullptr) return;
  {
    DeviceGuard g(P->device);
    cudaDeviceSynchronize();
    cudaFree(P->d_mem);
    if (P->d_lamb) cudaFree(P->d_lamb);
  }
  delete P;
}

int opt_plan_info(const opt_plan* P, int64_t* n_chunks, int64_t* total_numel, int64_t* workspace_bytes) {
  if (P == nullptr) return OPT_EINVAL;
  if (n_chunks) *n_chunks = P->n_chunks;
  if (total_numel) *total_numel = P->total_numel;
  if (workspace_bytes) *workspace_bytes = P->d_bytes;
  return OPT_OK;
}

const opt_norm_result* opt_plan_norm_buffer(const opt_plan* P) {
  return P ? P->d_result : nullptr;
}

int opt_grad_norm(opt_plan* P, double max_norm, opt_norm_result* d_out, opt_norm_result* h_out,
                  void* stream) {
  if (P == nullptr) return OPT_EINVAL;
  if (d_out != nullptr && ((uintptr_t)d_out & 7u)) return OPT_EALIGN;
  DeviceGuard g(P->device);
  if (!g.ok) return OPT_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  opt_norm_result* dst = d_out ? d_out : P->d_result;
  // one pass-1 launch per non-empty dtype bucket; its last CTA finishes
  cudaError_t e = launch_norm(P->d_chunks, P->bucket_begin, P->d_slots, P->d_done, max_norm, dst, s);
  if (e != cudaSuccess) return cuda_status(e);
  if (h_out != nullptr) {
    e = cudaMemcpyAsync(h_out, dst, sizeof(opt_norm_result), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    return h_out->status;
  }
  return OPT_OK;
}

static int do_step(opt_plan* P, const opt_hparams* hp, int64_t step, const opt_norm_result* d_norm,
                   void* stream, int algo) {
  if (P == nullptr || hp == nullptr) return OPT_EINVAL;
  if ((hp->flags & ~(OPT_STEP_RESET_STATES | OPT_STEP_DEVICE_COUNTER | OPT_STEP_WAIT_DRILL)) != 0)
    return OPT_EINVAL;
  const bool dev_step = (hp->flags & OPT_STEP_DEVICE_COUNTER) != 0;
  if (dev_step ? step != 0 : step < 1) return OPT_EINVAL;
  if (dev_step && P->combo != SC_F32) return OPT_EUNSUPPORTED;
  if (hp->rounding != OPT_ROUND_NEAREST && hp->rounding != OPT_ROUND_STOCHASTIC) return OPT_EINVAL;
  const bool drill = (hp->flags & OPT_STEP_WAIT_DRILL) != 0;
  if (drill && (algo != ALGO_ADAMW || !step_is_staged(P->combo, hp->rounding == OPT_ROUND_STOCHASTIC)))
    return OPT_EUNSUPPORTED;
  if (d_norm != nullptr && ((uintptr_t)d_norm & 7u)) return OPT_EALIGN;
  if (algo == ALGO_ADEMAMIX) {
    if (P->combo != SC_F32) return OPT_EUNSUPPORTED;
    if (!P->has_m2) return OPT_EINVAL;
  }
  StepArgs a;
  std::memset(&a, 0, sizeof a);
  // with the device counter the block's bias corrections are formed on the
  // device for the counter's next step; the rest is validated and formed here
  int st = opt_step_scalars_compute(hp, dev_step ? 1 : step, &a.sc);
  if (st != OPT_OK) return st;
  a.tensors = P->d_tensors;
  a.tiles = P->d_tiles;
  philox_round_keys(hp->seed, a.rk);
  a.neg_zero2 = kNegZero2;
  a.step32 = (uint32_t)step;
  a.d_norm = d_norm;
  a.unchanged = hp->count_unchanged ? P->d_unchanged : nullptr;
  a.reset = (hp->flags & OPT_STEP_RESET_STATES) ? 1 : 0;
  a.err = P->d_err;
  a.wait_ns = P->wait_ns;
  a.drill = drill ? 1 : 0;
  a.dyn = P->d_dyn;

  DeviceGuard g(P->device);
  if (!g.ok) return OPT_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (dev_step) {
    e = launch_step_scalars(a.sc, P->d_step, P->d_sc, s);
    a.d_sc = P->d_sc;
  }
  for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
    a.tile_begin = P->tile_begin[b];
    a.tile_end = P->tile_begin[b + 1];
    if (a.tile_end <= a.tile_begin) continue;
    const int dt = b == 0 ? OPT_F32 : OPT_BF16;
    const bool sr = hp->rounding == OPT_ROUND_STOCHASTIC;
    if (P->small_ok[b] && !dev_step && !drill) e = launch_step_small(dt, P->combo, algo, sr, a, P->small[b], s);
    else if (P->combo == SC_F32) e = launch_step_fp32_states(dt, algo, a, P->sm_count, s);
    else e = launch_step_lowp_states(dt, P->combo, sr, a, P->sm_count, s);
  }
  return cuda_status(e);
}

int opt_lamb_step(opt_plan* P, const opt_hparams* hp, int64_t step, float max_unorm,
                  const opt_norm_result* d_norm, void* stream) {
  if (P == nullptr || hp == nullptr || step < 1 || hp->flags != 0) return OPT_EINVAL;
  if (!(max_unorm >= 0.0f) || !std::isfinite(max_unorm)) return OPT_EINVAL;
  if (d_norm != nullptr && ((uintptr_t)d_norm & 7u)) return OPT_EALIGN;
  if (P->combo != SC_F32) return OPT_EUNSUPPORTED;
  StepArgs a;
  std::memset(&a, 0, sizeof a);
  int st = opt_step_scalars_compute(hp, step, &a.sc);
  if (st != OPT_OK) return st;
  a.tensors = P->d_tensors;
  a.tiles = P->d_tiles;
  a.d_norm = d_norm;
  a.err = P->d_err;
  a.dyn = P->d_dyn;
  DeviceGuard g(P->device);
  if (!g.ok) return OPT_ECUDA;
  cudaError_t e = cudaSuccess;
  if (P->d_lamb == nullptr && P->n > 0) {
    // segments of at most kLambSegTiles tiles, each tensor at least one
    std::vector<int32_t> seg_tensor, seg_count, tensor_seg0((size_t)P->n), tensor_nseg((size_t)P->n);
    std::vector<int64_t> seg_first;
    for (int32_t t = 0; t < P->n; ++t) {
      const int64_t first = P->tile_first[(size_t)t], count = P->tile_count[(size_t)t];
      const int64_t nseg = count > 0 ? (count + kLambSegTiles - 1) / kLambSegTiles : 1;
      tensor_seg0[(size_t)t] = (int32_t)seg_tensor.size();
      tensor_nseg[(size_t)t] = (int32_t)nseg;
      for (int64_t j = 0; j < nseg; ++j) {
        const int64_t left = count - j * kLambSegTiles;
        seg_tensor.push_back(t);
        seg_first.push_back(first + j * kLambSegTiles);
        seg_count.push_back((int32_t)(left < kLambSegTiles ? (left > 0 ? left : 0) : kLambSegTiles));
      }
    }
    const int64_t ns = (int64_t)seg_tensor.size();
    // per tile: two doubles; per segment: tensor, first tile, count, two
    // doubles; per tensor: first segment, segment count, ticket, ratio
    const int64_t off_st = align_up(16 * P->n_tiles, 256);
    const int64_t off_sf = align_up(off_st + 4 * ns, 256);
    const int64_t off_sc = align_up(off_sf + 8 * ns, 256);
    const int64_t off_ss = align_up(off_sc + 4 * ns, 256);
    const int64_t off_t0 = align_up(off_ss + 16 * ns, 256);
    const int64_t off_tn = align_up(off_t0 + 4 * (int64_t)P->n, 256);
    const int64_t off_tk = align_up(off_tn + 4 * (int64_t)P->n, 256);
    const int64_t off_r = align_up(off_tk + 4 * (int64_t)P->n, 256);
    const int64_t bytes = align_up(off_r + 4 * (int64_t)P->n, 256);
    e = cudaMalloc(&P->d_lamb, (size_t)bytes);
    if (e != cudaSuccess) { P->d_lamb = nullptr; return cuda_status(e); }
    char* base = static_cast<char*>(P->d_lamb);
    LambWork& w = P->lamb;
    w.tile_sums = base;
    w.seg_tensor = reinterpret_cast<const int32_t*>(base + off_st);
    w.seg_first = reinterpret_cast<const int64_t*>(base + off_sf);
    w.seg_count = reinterpret_cast<const int32_t*>(base + off_sc);
    w.seg_sums = base + off_ss;
    w.tensor_seg0 = reinterpret_cast<const int32_t*>(base + off_t0);
    w.tensor_nseg = reinterpret_cast<const int32_t*>(base + off_tn);
    w.tickets = reinterpret_cast<unsigned int*>(base + off_tk);
    w.ratio = reinterpret_cast<float*>(base + off_r);
    w.n_segs = (int)ns;
    auto up = [&](int64_t off, const void* src, size_t n) {
      return n == 0 ? cudaSuccess : cudaMemcpy(base + off, src, n, cudaMemcpyHostToDevice);
    };
    e = cudaMemset(base + off_tk, 0, 4 * (size_t)P->n);
    if (e == cudaSuccess) e = up(off_st, seg_tensor.data(), 4 * (size_t)ns);
    if (e == cudaSuccess) e = up(off_sf, seg_first.data(), 8 * (size_t)ns);
    if (e == cudaSuccess) e = up(off_sc, seg_count.data(), 4 * (size_t)ns);
    if (e == cudaSuccess) e = up(off_t0, tensor_seg0.data(), 4 * (size_t)P->n);
    if (e == cudaSuccess) e = up(off_tn, tensor_nseg.data(), 4 * (size_t)P->n);
    if (e != cudaSuccess) {
      cudaFree(P->d_lamb);
      P->d_lamb = nullptr;
      return cuda_status(e);
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int phase = 0; phase < 3 && e == cudaSuccess; ++phase) {
    for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
      if (phase == 1 && b == 1) break;               // the ratios cover every tensor at once
      a.tile_begin = P->tile_begin[b];
      a.tile_end = P->tile_begin[b + 1];
      e = launch_lamb(b == 0 ? OPT_F32 : OPT_BF16, a, P->lamb, max_unorm, P->sm_count, s, phase);
    }
  }
  return cuda_status(e);
}

int opt_adamw_step(opt_plan* P, const opt_hparams* hp, int64_t step, const opt_norm_result* d_norm,
                   void* stream) {
  return do_step(P, hp, step, d_norm, stream, ALGO_ADAMW);
}

int opt_ademamix_step(opt_plan* P, const opt_hparams* hp, int64_t step, const opt_norm_result* d_norm,
                      void* stream) {
  return do_step(P, hp, step, d_norm, stream, ALGO_ADEMAMIX);
}

int opt_unchanged_count(opt_plan* P, uint64_t* h_count, void* stream) {
  if (P == nullptr || h_count == nullptr) return OPT_EINVAL;
  DeviceGuard g(P->device);
  if (!g.ok) return OPT_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, P->d_unchanged, 8, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(P->d_unchanged, 0, 8, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_status(e);
  *h_count = v;
  return OPT_OK;
}

int opt_plan_set_step(opt_plan* P, int64_t next_step, void* stream) {
  if (P == nullptr || next_step < 1) return OPT_EINVAL;
  DeviceGuard g(P->device);
  if (!g.ok) return OPT_ECUDA;
  return cuda_status(launch_set_step(P->d_step, next_step - 1, static_cast<cudaStream_t>(stream)));
}

int opt_plan_status(opt_plan* P, int32_t* h_flags, void* stream) {
  if (P == nullptr || h_flags == nullptr) return OPT_EINVAL;
  DeviceGuard g(P->device);
  if (!g.ok) return OPT_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, P->d_err, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(P->d_err, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_status(e);
  *h_flags = v;
  return OPT_OK;
}

int opt_plan_set_wait_limit(opt_plan* P, uint64_t ns) {
  if (P == nullptr || ns > kMaxWaitNs) return OPT_EINVAL;
  P->wait_ns = ns;
  return OPT_OK;
}

int opt_grads_upload(opt_plan* P, const void* const* h_grad, void* stream) {
  if (P == nullptr || (P->n > 0 && h_grad == nullptr)) return OPT_EINVAL;
  for (int32_t i = 0; i < P->n; ++i)
    if (P->grad_bytes[(size_t)i] > 0 && h_grad[i] == nullptr) return OPT_EINVAL;
  DeviceGuard g(P->device);
  if (!g.ok) return OPT_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int32_t i = 0; i < P->n; ++i) {
    if (P->grad_bytes[(size_t)i] == 0) continue;
    cudaError_t e = cudaMemcpyAsync(P->grad_dev[(size_t)i], h_grad[i], (size_t)P->grad_bytes[(size_t)i],
                                    cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return OPT_OK;
}

int opt_encode(const float* d_in, void* d_out, int64_t n, int32_t dtype, int32_t rounding, uint64_t seed,
               uint32_t tensor_index, int64_t step, void* stream) {
  if (n < 0 || step < 0) return OPT_EINVAL;
  if (dtype != OPT_BF16 && dtype != OPT_E4M3 && dtype != OPT_E2M2) return OPT_EUNSUPPORTED;
  if (rounding != OPT_ROUND_NEAREST && rounding != OPT_ROUND_STOCHASTIC) return OPT_EINVAL;
  if (n == 0) return OPT_OK;
  if (d_in == nullptr || d_out == nullptr) return OPT_EINVAL;
  if (!aligned16(d_in) || !aligned16(d_out)) return OPT_EALIGN;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return OPT_ECUDA;
  return cuda_status(launch_encode(d_in, d_out, n, dtype, rounding == OPT_ROUND_STOCHASTIC,
                                   (uint32_t)seed, (uint32_t)(seed >> 32), tensor_index, (uint32_t)step,
                                   sms, static_cast<cudaStream_t>(stream)));
}

int opt_decode(const void* d_in, float* d_out, int64_t n, int32_t dtype, void* stream) {
  if (n < 0) return OPT_EINVAL;
  if (dtype != OPT_BF16 && dtype != OPT_E4M3 && dtype != OPT_E2M2) return OPT_EUNSUPPORTED;
  if (n == 0) return OPT_OK;
  if (d_in == nullptr || d_out == nullptr) return OPT_EINVAL;
  if (!aligned16(d_in) || !aligned16(d_out)) return OPT_EALIGN;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return OPT_ECUDA;
  return cuda_status(launch_decode(d_in, d_out, n, dtype, sms, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

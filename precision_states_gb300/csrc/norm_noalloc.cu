// norm_noalloc.cu -- opt_grad_norm_noalloc: the global gradient norm for
// callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not an option -- inside a
// framework whose caching allocator owns every byte of device memory and must
// not be bypassed, in a runtime with a fixed, pre-reserved memory budget, or
// at a point where a synchronising allocation would stall a pipeline.  Such a
// caller cannot build a plan (opt_plan_create allocates its workspace).
//
// How: every byte of scratch this call needs lives in one file-scope device
// array, g_noalloc_scratch, sized for at most OPT_NOALLOC_MAX_TENSORS tensors
// and OPT_NOALLOC_MAX_CHUNKS chunks.  Every GPU that loads the library holds
// it until the process exits.  Host code cannot use the array's name as a
// device address (in host code it names a host-side stand-in), so the first
// call on each device looks the address up with cudaGetSymbolAddress, with
// that device current, and caches it.  Each call then copies the caller's
// host arrays into the array (cudaMemcpyAsync, no staging buffer of ours),
// builds the chunk table on the device in the same order and with the same
// chunk sizes (chosen on the host from the sizes, as opt_chunk_table does)
// as opt_plan_create builds it on the host, and runs the same norm kernels
// as opt_grad_norm -- so the result is the same, bit for bit.
//
// Every call shares the array and overwrites the parts it reads before
// reading them -- all but the norm's completion counter, which the
// finishing CTA returns to 0 -- so nothing carries over from the previous
// call.  Two calls whose device work overlaps (different streams, or
// different host threads) race on the array.
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace psopt {
namespace {

constexpr int kMaxTensors = OPT_NOALLOC_MAX_TENSORS;
constexpr int64_t kMaxChunks = OPT_NOALLOC_MAX_CHUNKS;
constexpr int kPrepThreads = 1024;
constexpr int kPerThread = kMaxTensors / kPrepThreads;   // 8
static_assert(kMaxTensors % kPrepThreads == 0, "prep layout");

// scratch layout (byte offsets, each 256-aligned)
constexpr int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }
constexpr int64_t kOffGrad = 0;                                            // const void*[T]
constexpr int64_t kOffNumel = align256(kOffGrad + 8 * kMaxTensors);        // int64[T]
constexpr int64_t kOffDtype = align256(kOffNumel + 8 * kMaxTensors);       // int32[T]
constexpr int64_t kOffOrder = align256(kOffDtype + 4 * kMaxTensors);       // int32[T]
constexpr int64_t kOffBase = align256(kOffOrder + 4 * kMaxTensors);        // int64[T]: first chunk, in that order
constexpr int64_t kOffChunks = align256(kOffBase + 8 * kMaxTensors);       // NormChunk[C]
constexpr int64_t kOffSlots = align256(kOffChunks + 16 * kMaxChunks);      // NormSlot[2 * OPT_NORM_SLOTS]
constexpr int64_t kOffDone = align256(kOffSlots + 32 * 2 * OPT_NORM_SLOTS);    // uint32: completion counter
constexpr int64_t kScratchBytes = align256(kOffDone + 4);

static_assert(kScratchBytes == 4466432, "scratch size stated in opt.h");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch per device, looked up once per device.
constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

cudaError_t scratch_address(int device, unsigned char** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[device] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[device] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch_addr[device]);
  return cudaSuccess;
}

// One CTA: per-tensor chunk counts (chunks of ce0 elements in the FP32
// bucket, ce1 in the BF16 one), a stable bucket-major order (FP32 gradients
// first, then BF16, list order within a bucket), and each tensor's first
// chunk in that order.
__global__ void __launch_bounds__(kPrepThreads)
noalloc_prep_kernel(unsigned char* scratch, int n, int64_t ce0, int64_t ce1) {
  const int64_t* numel = reinterpret_cast<const int64_t*>(scratch + kOffNumel);
  const int32_t* dtype = reinterpret_cast<const int32_t*>(scratch + kOffDtype);
  int32_t* order = reinterpret_cast<int32_t*>(scratch + kOffOrder);
  int64_t* base = reinterpret_cast<int64_t*>(scratch + kOffBase);

  __shared__ int64_t s_chunks[2][kPrepThreads];   // per-thread chunk totals per bucket
  __shared__ int s_count[2][kPrepThreads];        // per-thread tensor counts per bucket
  const int tid = threadIdx.x;
  const int t0 = tid * kPerThread;                // this thread's tensors: t0 .. t0+7
  int64_t ch[2] = {0, 0};
  int cnt[2] = {0, 0};
  for (int k = 0; k < kPerThread; ++k) {
    const int t = t0 + k;
    if (t >= n) break;
    const int b = dtype[t] == OPT_BF16 ? 1 : 0;
    const int64_t ce = b ? ce1 : ce0;
    ch[b] += (numel[t] + ce - 1) / ce;
    cnt[b] += 1;
  }
  s_chunks[0][tid] = ch[0]; s_chunks[1][tid] = ch[1];
  s_count[0][tid] = cnt[0]; s_count[1][tid] = cnt[1];
  __syncthreads();
  // inclusive Hillis-Steele scans over threads (both buckets)
  for (int off = 1; off < kPrepThreads; off <<= 1) {
    int64_t a0 = 0, a1 = 0;
    int c0 = 0, c1 = 0;
    if (tid >= off) {
      a0 = s_chunks[0][tid - off]; a1 = s_chunks[1][tid - off];
      c0 = s_count[0][tid - off]; c1 = s_count[1][tid - off];
    }
    __syncthreads();
    s_chunks[0][tid] += a0; s_chunks[1][tid] += a1;
    s_count[0][tid] += c0; s_count[1][tid] += c1;
    __syncthreads();
  }
  const int64_t total0 = s_chunks[0][kPrepThreads - 1];
  const int n0 = s_count[0][kPrepThreads - 1];
  int64_t next[2] = {s_chunks[0][tid] - ch[0], total0 + s_chunks[1][tid] - ch[1]};
  int pos[2] = {s_count[0][tid] - cnt[0], n0 + s_count[1][tid] - cnt[1]};
  for (int k = 0; k < kPerThread; ++k) {
    const int t = t0 + k;
    if (t >= n) break;
    const int b = dtype[t] == OPT_BF16 ? 1 : 0;
    const int64_t ce = b ? ce1 : ce0;
    order[pos[b]] = t;
    base[pos[b]] = next[b];
    pos[b] += 1;
    next[b] += (numel[t] + ce - 1) / ce;
  }
}

// One thread per chunk: find its tensor (last position whose first chunk is
// <= c, by binary search over the bucket-major order) and write the entry
// with the chunk's first gradient element resolved.
__global__ void noalloc_fill_kernel(unsigned char* scratch, int n, int64_t total, int64_t ce0, int64_t ce1) {
  const void* const* grad = reinterpret_cast<const void* const*>(scratch + kOffGrad);
  const int64_t* numel = reinterpret_cast<const int64_t*>(scratch + kOffNumel);
  const int32_t* dtype = reinterpret_cast<const int32_t*>(scratch + kOffDtype);
  const int32_t* order = reinterpret_cast<const int32_t*>(scratch + kOffOrder);
  const int64_t* base = reinterpret_cast<const int64_t*>(scratch + kOffBase);
  NormChunk* chunks = reinterpret_cast<NormChunk*>(scratch + kOffChunks);
  for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < total;
       c += (int64_t)gridDim.x * blockDim.x) {
    int lo = 0, hi = n;            // first position with base > c
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (base[mid] <= c) lo = mid + 1;
      else hi = mid;
    }
    const int t = order[lo - 1];
    const int64_t ce = dtype[t] == OPT_BF16 ? ce1 : ce0;
    const int64_t start = (c - base[lo - 1]) * ce;
    const int64_t left = numel[t] - start;
    NormChunk e;
    e.ptr = static_cast<const char*>(grad[t]) + start * (dtype[t] == OPT_BF16 ? 2 : 4);
    e.len = (uint32_t)(left < ce ? left : ce);
    e.pad = 0;
    chunks[c] = e;
  }
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return OPT_OK;
  return e == cudaErrorMemoryAllocation ? OPT_ENOMEM : OPT_ECUDA;
}

}  // namespace
}  // namespace psopt

using namespace psopt;

extern "C" int opt_grad_norm_noalloc(int32_t n, const int64_t* numel, const void* const* grad,
                                     const int32_t* grad_dtype, double max_norm, opt_norm_result* d_out,
                                     void* stream) {
  // ---- host-side validation, before any CUDA call
  if (n < 0 || d_out == nullptr) return OPT_EINVAL;
  if ((uintptr_t)d_out & 7u) return OPT_EALIGN;
  if (n > kMaxTensors) return OPT_ELIMIT;
  if (n > 0 && (numel == nullptr || grad == nullptr || grad_dtype == nullptr)) return OPT_EINVAL;
  for (int32_t i = 0; i < n; ++i) {
    if (numel[i] < 0) return OPT_EINVAL;
    if (grad_dtype[i] != OPT_F32 && grad_dtype[i] != OPT_BF16) return OPT_EUNSUPPORTED;
    if (numel[i] > 0 && grad[i] == nullptr) return OPT_EINVAL;
    if (grad[i] != nullptr && ((uintptr_t)grad[i] & 15u)) return OPT_EALIGN;
  }
  int64_t ce[2];
  for (int b = 0; b < 2; ++b) {
    ce[b] = norm_chunk_elems(n, numel, grad_dtype, b);
    if (ce[b] < 0) return (int)ce[b];
  }
  int64_t bucket[2] = {0, 0};
  for (int32_t i = 0; i < n; ++i) {
    const int b = grad_dtype[i] == OPT_BF16 ? 1 : 0;
    bucket[b] += (numel[i] + ce[b] - 1) / ce[b];
    if (bucket[0] + bucket[1] > kMaxChunks) return OPT_ELIMIT;
  }
  const int64_t total = bucket[0] + bucket[1];

  int dev = 0;
  unsigned char* scratch = nullptr;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = scratch_address(dev, &scratch);
  if (e != cudaSuccess) return cuda_status(e);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (n > 0) {
    e = cudaMemcpyAsync(scratch + kOffGrad, grad, sizeof(void*) * (size_t)n, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(scratch + kOffNumel, numel, sizeof(int64_t) * (size_t)n, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(scratch + kOffDtype, grad_dtype, sizeof(int32_t) * (size_t)n, cudaMemcpyHostToDevice,
                          s);
    if (e != cudaSuccess) return cuda_status(e);
    noalloc_prep_kernel<<<1, kPrepThreads, 0, s>>>(scratch, n, ce[0], ce[1]);
    if (total > 0) {
      const int64_t want = (total + 255) / 256;
      noalloc_fill_kernel<<<(int)(want < 1024 ? want : 1024), 256, 0, s>>>(scratch, n, total, ce[0], ce[1]);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
  }

  const NormChunk* chunks = reinterpret_cast<const NormChunk*>(scratch + kOffChunks);
  NormSlot* slots = reinterpret_cast<NormSlot*>(scratch + kOffSlots);
  unsigned int* done = reinterpret_cast<unsigned int*>(scratch + kOffDone);
  const int64_t begin[3] = {0, bucket[0], total};
  e = launch_norm(chunks, begin, slots, done, max_norm, d_out, s);
  return cuda_status(e);
}

"""GPU parity of the standalone state codecs (opt_encode / opt_decode) with
the oracle: bit-exact codes for every format and rounding mode, including
subnormals, ties, saturation, NaN/Inf and ragged lengths."""
import functools

import numpy as np
import pytest
import torch

import oracle
import precision_states_gb300 as ps

pytestmark = pytest.mark.gpu

ENC = {"bf16": oracle.bf16_encode, "e4m3": oracle.e4m3_encode, "e2m2": oracle.e2m2_encode}


@functools.lru_cache(maxsize=1)
def cached_values(n, seed):
    """sample_values, kept for the next parameter set of the same size (the
    inputs are only read)."""
    return sample_values(n, seed)


def sample_values(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n) * np.exp(rng.uniform(-25, 12, n))
    x = x.astype(np.float32)
    # the E4M3 / E2M2 ranges, their subnormals and exact grid points and midpoints
    x[: n // 4] = (rng.uniform(0, 500, n // 4) * rng.choice([1e-3, 1e-2, 1, 2 ** -8], n // 4)).astype(np.float32)
    specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 448.0, 464.0, 480.0, 7.0, 7.5, 0.125,
                         0.375, 2 ** -9, 2 ** -10, 3 * 2 ** -11, 1e-40, -1e-40, 3.4e38, -7.25,
                         1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8], np.float32)
    if n >= 2 * len(specials):
        x[-len(specials):] = specials
    return x


def enc_size(dtype, n):
    return ps.state_nbytes(dtype, n)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3", "e2m2"])
@pytest.mark.parametrize("rounding", ["nearest", "stochastic"])
@pytest.mark.parametrize("n", [40001, 9, 8])
def test_encode_matches_oracle(dtype, rounding, n):
    x = sample_values(n, seed=n + len(dtype))
    seed, step, tidx = 0xDEADBEEF12345678, 17, 5
    d_in = torch.from_numpy(x).cuda()
    d_out = torch.full((enc_size(dtype, n),), 0xAB, dtype=torch.uint8, device="cuda")
    ps.opt_encode(d_in, d_out, dtype, rounding=rounding, seed=seed, tensor_index=tidx, step=step)
    torch.cuda.synchronize()
    got = d_out.cpu().numpy()
    sr = rounding == "stochastic"
    want = []
    for i, xv in enumerate(x):
        r = oracle.cast_draw(seed, step, tidx, i) if sr else 0
        want.append(ENC[dtype](float(xv), sr, r))
    want = np.array(want, dtype=np.uint32)
    if dtype == "bf16":
        g = got.view(np.uint16).astype(np.uint32)
    elif dtype == "e4m3":
        g = got.astype(np.uint32)
    else:
        g = np.stack([got & 0xF, got >> 4], axis=1).ravel()[:n].astype(np.uint32)
        if n % 2:
            assert (got[-1] >> 4) == 0, "unused high nibble must be 0"
    # NaN: BF16 keeps a quiet NaN with the input's top payload bits
    mism = np.nonzero(g != want)[0]
    assert mism.size == 0, f"{mism.size} mismatches, first at {mism[0]}: x={x[mism[0]]!r} got={g[mism[0]]:#x} want={want[mism[0]]:#x}"


@pytest.mark.parametrize("dtype", ["bf16", "e4m3", "e2m2"])
def test_decode_all_codes(dtype):
    if dtype == "bf16":
        codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
        n = codes.size
        raw = codes.view(np.uint8)
        want = np.array([oracle.bf16_decode(int(c)) for c in codes], np.float32)
    elif dtype == "e4m3":
        raw = np.arange(256, dtype=np.uint8)
        n = 256
        want = np.array([oracle.e4m3_decode(int(c)) for c in raw], np.float32)
    else:
        c = np.arange(16, dtype=np.uint8)
        c = np.concatenate([c, c[::-1], c[:7]])     # odd length
        n = c.size
        raw = np.zeros((n + 1) // 2, np.uint8)
        for i, v in enumerate(c):
            raw[i // 2] |= v << (4 * (i & 1))
        want = np.array([oracle.e2m2_decode(int(v)) for v in c], np.float32)
    d_in = torch.from_numpy(raw.copy()).cuda()
    d_out = torch.empty(n, dtype=torch.float32, device="cuda")
    ps.opt_decode(d_in, d_out, n, dtype)
    got = d_out.cpu().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def _codes_of(dtype, raw, n):
    if dtype == "bf16":
        return raw.view(np.uint16).astype(np.uint32)
    if dtype == "e4m3":
        return raw.astype(np.uint32)
    return np.stack([raw & 0xF, raw >> 4], axis=1).ravel()[:n].astype(np.uint32)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3", "e2m2"])
@pytest.mark.parametrize("rounding", ["nearest", "stochastic"])
@pytest.mark.parametrize("n", [6_000_003, (1 << 28) + 12])
def test_encode_many_grid_strides_sampled(dtype, rounding, n):
    """6,000,003 elements: several grid strides of two-group iterations, a
    lone last group for some threads and a 3-element tail; and 2^28 + 12, the
    size `bench.py --cast` times, in the same launch.  30,000 sampled
    positions plus the first and last 64 against the oracle."""
    x = cached_values(n, 77)
    seed, step, tidx = 0x0123456789ABCDEF, 1000, 290
    d_in = torch.from_numpy(x).cuda()
    d_out = torch.zeros((enc_size(dtype, n),), dtype=torch.uint8, device="cuda")
    ps.opt_encode(d_in, d_out, dtype, rounding=rounding, seed=seed, tensor_index=tidx, step=step)
    torch.cuda.synchronize()
    g = _codes_of(dtype, d_out.cpu().numpy(), n)
    rng = np.random.default_rng(5)
    idx = np.unique(np.concatenate([rng.integers(0, n, 30000), np.arange(64), np.arange(n - 64, n)]))
    sr = rounding == "stochastic"
    for i in idx:
        r = oracle.cast_draw(seed, step, tidx, int(i)) if sr else 0
        want = ENC[dtype](float(x[i]), sr, r)
        assert g[i] == want, f"element {i}: x={x[i]!r} got={g[i]:#x} want={want:#x}"


@pytest.mark.parametrize("dtype", ["bf16", "e4m3", "e2m2"])
def test_decode_random_codes_large(dtype):
    """1,000,003 random codes decoded on the GPU equal the oracle's decode of
    each code (through a table of all codes)."""
    n = 1_000_003
    rng = np.random.default_rng(11)
    ncodes = {"bf16": 1 << 16, "e4m3": 256, "e2m2": 16}[dtype]
    dec = {"bf16": oracle.bf16_decode, "e4m3": oracle.e4m3_decode, "e2m2": oracle.e2m2_decode}[dtype]
    table = np.array([dec(c) for c in range(ncodes)], np.float32)
    codes = rng.integers(0, ncodes, n)
    if dtype == "bf16":
        raw = codes.astype(np.uint16).view(np.uint8)
    elif dtype == "e4m3":
        raw = codes.astype(np.uint8)
    else:
        c = np.concatenate([codes, [0]]).astype(np.uint8)
        raw = (c[0::2] | (c[1::2] << 4)).astype(np.uint8)
    d_in = torch.from_numpy(raw.copy()).cuda()
    d_out = torch.empty(n, dtype=torch.float32, device="cuda")
    ps.opt_decode(d_in, d_out, n, dtype)
    got = d_out.cpu().numpy()
    want = table[codes]
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_encode_draws_independent_of_launch_shape():
    """The draw is tied to the element ("When Small Updates Disappear",
    sec. 7.3): encoding a prefix gives the same codes as encoding the whole."""
    x = sample_values(100000, 3)
    d = torch.from_numpy(x).cuda()
    full = torch.empty(100000 * 2, dtype=torch.uint8, device="cuda")
    part = torch.empty(77777 * 2 + 14, dtype=torch.uint8, device="cuda")
    ps.opt_encode(d, full, "bf16", rounding="stochastic", seed=9, tensor_index=1, step=3)
    ps.opt_encode(d[:77777], part, "bf16", rounding="stochastic", seed=9, tensor_index=1, step=3)
    torch.cuda.synchronize()
    assert torch.equal(full[: 77777 * 2], part[: 77777 * 2])

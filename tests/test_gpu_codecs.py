"""GPU parity of the standalone state codecs (opt_encode / opt_decode) with
the oracle: bit-exact codes for every format and rounding mode, including
subnormals, ties, saturation, NaN/Inf and ragged lengths."""
import numpy as np
import pytest
import torch

import oracle
import precision_states_gb300 as ps

pytestmark = pytest.mark.gpu

ENC = {"bf16": oracle.bf16_encode, "e4m3": oracle.e4m3_encode, "e2m2": oracle.e2m2_encode}


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
        r = oracle.draws(seed, step, tidx, i)[1] if sr else 0
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

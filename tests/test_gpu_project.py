"""GPU parity of the direction projection u = normalize(W_u k_raw) (vla_project_u).

README "VLA v3" item 2 forms the scan's directions as u_t = normalize(W_u k_t^raw).
The float64 oracle (oracle.project_u, pinned by closed forms) on the same rounded
keys and float32 weights, rounded to the I/O dtype, is the reference.

The kernel's arithmetic: float32 keys go through tcgen05 kind::tf32 with keys and W
split into tf32 high and low parts (about 2^-21 relative); bfloat16 keys (exact in
bf16) go through kind::f16 with W carried as three bfloat16 terms w1 + w2 + w3
(about 24 bits), accumulated in float32.  The tolerance follows: a float32 dot
product of length d errs by at most about d * 2^-24 times the sum of its terms'
sizes, a few 1e-6 in absolute terms on a unit vector, and a bfloat16 result may
round to the neighbour of the rounded float64 value (one unit in the last place).
Because one ulp would also hide a lost W term (w1 alone is good to 2^-9), the bf16
tests also require that at least 99.9 % of the outputs equal the rounded float64
value exactly: with all three terms about 0.01 % differ, without w3 about 0.25 %,
without w2 and w3 about 40 %.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from _util import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    import sherman_morrison_inverse_gb300 as vla
    vla.load_library()


def _ref(k, W, dtype):
    u = oracle.project_u(k.reshape(-1, k.shape[-1]), W)
    return torch.from_numpy(u).to(dtype).double().numpy().reshape(*k.shape[:-1], W.shape[0], k.shape[-1])


def _check(got, ref, dtype):
    d = got.shape[-1]
    fp32 = d * 2.0 ** -24 * 4        # the float32 summation bound on a unit vector (|W|, |k| of order 1)
    diff = np.abs(got - ref)
    if dtype == torch.bfloat16:   # plus one bf16 ulp of the reference value
        bound = np.abs(ref) * 2.0 ** -7 + fp32
    else:
        bound = np.full_like(ref, fp32)
    assert np.all(diff <= bound), float(np.max(diff / bound))
    if dtype == torch.bfloat16:
        exact = float(np.mean(got == ref))
        assert exact >= 0.999, f"only {exact:.5f} of the bf16 outputs equal the rounded float64 value"


@pytest.mark.parametrize("d,r,dtype,n", [(16, 1, torch.float32, 300), (64, 1, torch.bfloat16, 1000),
                                         (64, 4, torch.float32, 257), (128, 1, torch.bfloat16, 129),
                                         (128, 4, torch.float32, 77)])
def test_projection_matches_oracle(d, r, dtype, n):
    import sherman_morrison_inverse_gb300 as vla
    g = np.random.default_rng([d, r, n])
    k = torch.from_numpy(g.normal(size=(n, d))).to(dtype)
    W = torch.from_numpy(g.normal(size=(r, d, d)) / np.sqrt(d)).float()
    u = vla.project_u(k.cuda(), W.cuda()).double().cpu().numpy()
    _check(u, _ref(k.double().numpy(), W.double().numpy(), dtype), dtype)


def test_projection_of_the_recall_workload_keys():
    """The recall workload's keys and W_u ([B, H, T, d] keys, B H T tokens), all tokens."""
    import sherman_morrison_inverse_gb300 as vla
    w = workloads.get(2)
    x = workloads.make_inputs(w, pairs=[0, 1, 2], T=4096)
    k = x["k"]   # [3, T, d] bf16
    u = vla.project_u(k.cuda(), x["Wu"].cuda()).double().cpu().numpy()
    _check(u, _ref(k.double().numpy(), x["Wu"].double().numpy(), torch.bfloat16), torch.bfloat16)


def test_zero_keys_give_zero_directions_and_n0_is_a_no_op():
    import sherman_morrison_inverse_gb300 as vla
    k = torch.zeros((5, 64), device="cuda")
    W = torch.eye(64, device="cuda")[None]
    assert torch.count_nonzero(vla.project_u(k, W)) == 0
    empty = torch.empty((0, 64), device="cuda")
    assert vla.project_u(empty, W).shape == (0, 1, 64)


def test_projection_rejects_unbuilt_width():
    import sherman_morrison_inverse_gb300 as vla
    with pytest.raises(vla.VlaError, match="UNSUPPORTED"):
        vla.project_u(torch.zeros((4, 32), device="cuda"), torch.zeros((1, 32, 32), device="cuda"))


def test_projection_rejects_misaligned_pointers():
    """Rows move as 16-byte vectors: a key tensor that starts 2 bytes into its buffer is refused."""
    import sherman_morrison_inverse_gb300 as vla
    buf = torch.zeros(4 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    k = buf[1:1 + 4 * 64].view(4, 64)
    assert k.data_ptr() % 16 != 0
    with pytest.raises(vla.VlaError, match="INVALID_ARG"):
        vla.project_u(k, torch.eye(64, device="cuda")[None])


def test_projection_grid_stride_covers_every_token():
    """More tokens than one pass of the grid (4 CTAs of 128 threads per SM): every row is
    written, including the ragged end."""
    import sherman_morrison_inverse_gb300 as vla
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = 4 * 128 * sms * 2 + 37
    g = np.random.default_rng(5)
    k = torch.from_numpy(g.normal(size=(n, 16))).float()
    W = torch.from_numpy(g.normal(size=(2, 16, 16)) / 4.0).float()
    u = vla.project_u(k.cuda(), W.cuda()).double().cpu().numpy()
    _check(u, _ref(k.double().numpy(), W.double().numpy(), torch.float32), torch.float32)


@pytest.mark.parametrize("d", [16, 64, 128])
@pytest.mark.parametrize("r", [1, 4])
def test_bf16_projection_several_tiles_per_cta(d, r):
    """bfloat16 keys with many tiles per CTA: the TMA form's persistent grid (one CTA per SM)
    cycles its key stages and both accumulators many times, the register form (d = 128,
    r = 4: 8 CTAs of 128 tokens per SM) runs its main loop over at least two tiles, and the
    last tile is ragged.  The outputs are compared on a sample of tokens: the first and last
    tiles, the second and third tile of the first CTAs, and random ones."""
    import sherman_morrison_inverse_gb300 as vla
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    grid = 8 * sms
    n = 2 * grid * 128 + 2 * 128 + 37
    g = np.random.default_rng([d, r, 7])
    k = torch.from_numpy(g.normal(size=(n, d)).astype(np.float32)).to(torch.bfloat16)
    W = torch.from_numpy(g.normal(size=(r, d, d)) / np.sqrt(d)).float()
    u = vla.project_u(k.cuda(), W.cuda()).cpu()   # the sample is taken on the host
    idx = np.unique(np.concatenate([
        np.arange(0, 512), np.arange(n - 512, n),
        np.arange(grid * 128, grid * 128 + 3 * 128),          # CTAs 0..2, second tile
        np.arange(2 * grid * 128, n),                         # CTAs 0..2, third tile (the ragged end)
        g.integers(0, n, size=16384)]))
    assert idx.min() >= 0 and idx.max() < n
    got = u[torch.from_numpy(idx)].double().numpy()
    ref = _ref(k[torch.from_numpy(idx)].double().numpy(), W.double().numpy(), torch.bfloat16)
    _check(got, ref, torch.bfloat16)


@pytest.mark.parametrize("d,r,n", [(64, 1, 1), (64, 1, 127), (64, 1, 128), (64, 2, 129), (64, 3, 5000),
                                   (64, 4, 300), (64, 5, 200), (64, 5, 40000), (64, 8, 150), (16, 1, 40),
                                   (16, 3, 1000), (16, 5, 777), (16, 8, 129), (128, 1, 1000), (128, 2, 300),
                                   (128, 3, 130)])
def test_bf16_projection_every_rank_count_and_no_write_past_the_end(d, r, n):
    """bfloat16 keys for rank counts 1..8: the r weight sets stacked into one product of
    N = r d columns (d = 16 up to N = 128, d = 64 up to r = 4), two rank groups on one key
    tile (d = 64, r = 5: N = 256 and 64), and beyond what shared memory holds (d = 64 with
    r = 8, d = 128 with r > 1) the one-rank-at-a-time form; n below, at and just past one
    128-token tile, and many tiles per CTA.  Output rows past n in the caller's buffer keep
    their contents (the tensor stores clip the ragged last tile)."""
    import sherman_morrison_inverse_gb300 as vla
    g = np.random.default_rng([d, r, n, 11])
    k = torch.from_numpy(g.normal(size=(n, d)).astype(np.float32)).to(torch.bfloat16)
    W = torch.from_numpy(g.normal(size=(r, d, d)) / np.sqrt(d)).float()
    sentinel = 7.0
    ubuf = torch.full((n + 130, r, d), sentinel, dtype=torch.bfloat16, device="cuda")
    u = ubuf[:n]
    vla.project_u(k.cuda(), W.cuda(), u)
    host = ubuf.cpu()
    assert torch.all(host[n:] == sentinel), "rows past n were written"
    _check(host[:n].double().numpy(), _ref(k.double().numpy(), W.double().numpy(), torch.bfloat16), torch.bfloat16)

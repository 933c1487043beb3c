"""GPU parity of fa_fwd_f32x3 (fp32 on the tensor cores, three TF32
products per matrix product) against the fp64 oracle.

Tolerance: the fp32 path's 1e-5 on O and LSE (the fp32 check of
"Module 08: FlashAttention and Memory-Efficient Kernels", Code Step 4). The
split keeps about 22 significant bits of every product (the dropped lo*lo
term and the TF32 truncation of lo are each ~2^-22 of it), so for unit-scale
inputs the score error is ~2^-22 * scale * sum_d |q_d k_d| (~2e-6 at D = 128)
and O inherits it relatively, an order of magnitude inside the bound.
"""

import math

import numpy as np
import pytest

from oracle import attention
from flashattention_fa_fwd_gb300.inputs import WORKLOADS, make_inputs
from parity import check_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import flashattention_fa_fwd_gb300 as fa

    fa.load_library()


def run_x3(q, k, v, scale, causal):
    import torch

    import flashattention_fa_fwd_gb300 as fa

    dev = "cuda"
    qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev) for x in (q, k, v))
    B, H, M, D = qt.shape
    o = torch.full((B, H, M, D), float("nan"), device=dev)
    lse = torch.full((B, H, M), float("nan"), device=dev)
    fa.fa_fwd_f32x3(qt, kt, vt, o, lse, scale, causal)
    st = fa.fa_get_device_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return o.cpu().numpy(), lse.cpu().numpy()


def _rand(shape, seed, sigma=1.0):
    return np.random.default_rng(seed).standard_normal(shape, dtype=np.float32) * np.float32(sigma)


def test_f32x3_single_head_workload():
    w = WORKLOADS["f32_single_head_m256_n512_d64"]
    q, k, v = make_inputs(w)
    o, lse = run_x3(q, k, v, w.scale, w.causal)
    o_ref, lse_ref = attention(q, k, v, w.scale, w.causal)
    err = check_f32(o, lse, o_ref, lse_ref, w.name)
    assert err <= 5e-6, f"{w.name}: O max err {err:.3e}"


@pytest.mark.parametrize("D", [32, 64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("M,N", [(300, 700), (257, 129), (128, 128), (1, 200), (200, 1), (130, 33)])
def test_f32x3_shapes(D, causal, M, N):
    q, k, v = (_rand((1, 2, r, D), 7 * M + 3 * N + D + i) for i, r in enumerate((M, N, N)))
    o, lse = run_x3(q, k, v, 1 / math.sqrt(D), causal)
    o_ref, lse_ref = attention(q, k, v, 1 / math.sqrt(D), causal)
    check_f32(o, lse, o_ref, lse_ref, f"f32x3 {M}x{N}x{D} causal={causal}")


def split_error_bound(q, k, v, scale):
    """Worst-case error of the three-product split, for inputs whose scores
    are far from unit scale. Per term q_d k_d the split drops lo_q lo_k
    (<= 2^-22 |q_d k_d|, since |lo| <= 2^-11 |x|) and the tensor core
    truncates each lo to TF32 in the two cross terms (<= 2^-21 |q_d k_d|
    each): 1.25 * 2^-20 |q_d k_d| in all. So a scaled score is off by at most
    ds = 1.25 * 2^-20 * A, A = max_ij scale * sum_d |q_id| |k_jd|; LSE moves
    by at most ds and O = sum_j P_j V_j / sum_j P_j by at most
    ds * max_j |V_j - O| <= 2 ds max |V|. The 1e-5 of the fp32 check is
    added for the rest of the fp32 arithmetic."""
    aq = np.abs(q.astype(np.float64)).reshape(-1, *q.shape[-2:])
    ak = np.abs(k.astype(np.float64)).reshape(-1, *k.shape[-2:])
    A = max(float((aq[h] @ ak[h].T).max()) for h in range(aq.shape[0])) * scale
    ds = 1.25 * 2.0 ** -20 * A
    return 1e-5 + 2.0 * ds * float(np.abs(v).max()), 1e-5 + ds


def test_f32x3_batched_heads_and_large_logits():
    """Several (b, h) pairs and peaked softmax rows (scores with a standard
    deviation of 9): the max moves between key blocks and the rare rescale
    runs. Scores this large are outside the unit-scale regime of the 1e-5
    check; the bound is the split's worst case (split_error_bound)."""
    q = _rand((2, 3, 333, 128), 1, 3.0)
    k = _rand((2, 3, 517, 128), 2, 3.0)
    v = _rand((2, 3, 517, 128), 3)
    scale = 1 / math.sqrt(128)
    o_tol, lse_tol = split_error_bound(q, k, v, scale)
    for causal in (False, True):
        o, lse = run_x3(q, k, v, scale, causal)
        o_ref, lse_ref = attention(q, k, v, scale, causal)
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
        err = np.abs(o - o_ref).max()
        lerr = np.abs(lse - lse_ref).max()
        assert err <= o_tol, f"large logits causal={causal}: O max err {err:.3e} > {o_tol:.3e}"
        assert lerr <= lse_tol, f"large logits causal={causal}: LSE max err {lerr:.3e} > {lse_tol:.3e}"


def test_f32x3_row_max_rises_across_blocks():
    """Scores that grow with the key index, so every block raises every
    row's max by more than the rescale threshold."""
    M, N, D = 160, 256, 64
    q = np.ones((1, 1, M, D), np.float32) * np.float32(0.25)
    k = (np.arange(N, dtype=np.float32)[:, None] * np.float32(0.05) * np.ones((1, D), np.float32))[None, None]
    v = _rand((1, 1, N, D), 5)
    o, lse = run_x3(q, k, v, 1.0, False)
    o_ref, lse_ref = attention(q, k, v, 1.0, False)
    check_f32(o, lse, o_ref, lse_ref, "rising max")


def test_f32x3_worked_example_padded():
    """Scores [1, 2, 3], values [10, 20, 30] ("FlashAttention in Triton",
    worked example), padded to D = 32 with zeros: 25.7521038."""
    q = np.zeros((1, 1, 1, 32), np.float32)
    k = np.zeros((1, 1, 3, 32), np.float32)
    v = np.zeros((1, 1, 3, 32), np.float32)
    q[..., 0] = 1.0
    k[0, 0, :, 0] = [1.0, 2.0, 3.0]
    v[0, 0, :, 0] = [10.0, 20.0, 30.0]
    o, lse = run_x3(q, k, v, 1.0, False)
    assert abs(o[0, 0, 0, 0] - 25.7521038) <= 1e-5
    assert np.all(o[0, 0, 0, 1:] == 0.0)


def test_f32x3_empty_keys():
    """N = 0: O = 0 and LSE = -inf (no workspace needed)."""
    q = _rand((1, 2, 70, 64), 9)
    k = np.zeros((1, 2, 0, 64), np.float32)
    o, lse = run_x3(q, k, k, 0.125, False)
    assert np.all(o == 0.0) and np.all(np.isneginf(lse))


def test_f32x3_matches_exact_fp32_path_and_is_deterministic():
    import torch

    import flashattention_fa_fwd_gb300 as fa

    q, k, v = (torch.randn(2, 4, 700, 64, device="cuda", generator=torch.Generator("cuda").manual_seed(s))
               for s in (1, 2, 3))
    o1, o2, oe = (torch.empty_like(q) for _ in range(3))
    l1, l2, le = (torch.empty(2, 4, 700, device="cuda") for _ in range(3))
    fa.fa_fwd_f32x3(q, k, v, o1, l1, 0.125, True)
    fa.fa_fwd_f32x3(q, k, v, o2, l2, 0.125, True)
    fa.fa_fwd_f32(q, k, v, oe, le, 0.125, True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert (o1 - oe).abs().max().item() <= 1e-5
    assert (l1 - le).abs().max().item() <= 1e-5


@pytest.mark.parametrize("name,path,heads", [("f32_causal_b8_h32_s4096_d128", "x3", (0, 131, 255)),
                                             ("f32_gpt2m_b64_h16_s1024_d64", "x3", (0, 517, 1023)),
                                             ("f32_gpt2m_b64_h16_s1024_d64", "ieee", (0, 1023))])
def test_f32_full_size_sampled_rows(name, path, heads):
    """A whole fp32 benchmark workload on the GPU in the benchmark's launch
    shape (the tensor-core path, or the exact one), checked on 256 sampled
    rows of sampled heads against the oracle at the fp32 bound, and finite
    everywhere."""
    import torch

    import flashattention_fa_fwd_gb300 as fa
    from oracle import attention_rows
    from flashattention_fa_fwd_gb300.inputs import head_tensor, sample_rows

    w = WORKLOADS[name]
    q, k, v = make_inputs(w)
    tq, tk, tv = (torch.from_numpy(x).cuda() for x in (q, k, v))
    del q, k, v
    o = torch.empty_like(tq)
    lse = torch.empty(w.B, w.H, w.M, device="cuda")
    (fa.fa_fwd_f32x3 if path == "x3" else fa.fa_fwd_f32)(tq, tk, tv, o, lse, w.scale, w.causal)
    assert fa.fa_get_device_status() == fa.FA_OK
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    o_np, lse_np = o.cpu().numpy(), lse.cpu().numpy()
    for bh in heads:
        b, h = divmod(bh, w.H)
        rows = sample_rows(w.wid, bh, w.M, 256)
        qh, kh, vh = (head_tensor(w.wid, t, bh, r, w.D, 1.0, w.dtype) for t, r in ((0, w.M), (1, w.N), (2, w.N)))
        o_ref, lse_ref = attention_rows(qh, kh, vh, w.scale, w.causal, rows)
        check_f32(o_np[b, h, rows], lse_np[b, h, rows], o_ref, lse_ref, f"{name} {path} head {bh}")

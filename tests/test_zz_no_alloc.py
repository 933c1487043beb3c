"""fa_fwd_noalloc: the bf16 forward for callers that cannot allocate device
memory (their own memory pool owns the GPU, they must avoid the device-wide
synchronisation a cudaMalloc can cause, or they run under a fixed memory
quota). It keeps the kernel's scratch in a static device array instead of a
cudaMalloc'd buffer; its results must equal fa_fwd's.

This file is collected last on purpose, and it runs the same whether it is
alone in a fresh process or after every other test.
"""

import math

import numpy as np
import pytest

from parity import check_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import flashattention_fa_fwd_gb300 as fa

    fa.load_library()
    return fa


def _problem(torch, seed, B, H, M, N, D):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn(B, H, M, D, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(B, H, N, D, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(B, H, N, D, device="cuda", generator=g).to(torch.bfloat16)
    return q, k, v


def test_noalloc_matches_fa_fwd_on_two_calls_in_a_row(fa):
    import torch

    cases = [(11, 2, 3, 700, 900, 128, True), (12, 1, 4, 300, 1000, 64, False), (13, 2, 2, 333, 517, 96, False)]
    probs, refs, outs = [], [], []
    for seed, B, H, M, N, D, causal in cases:
        q, k, v = _problem(torch, seed, B, H, M, N, D)
        o_ref = torch.empty_like(q)
        l_ref = torch.empty(B, H, M, device="cuda")
        fa.fa_fwd(q, k, v, o_ref, l_ref, 1 / math.sqrt(D), causal)
        probs.append((q, k, v, B, H, M, N, D, causal))
        refs.append((o_ref, l_ref))
        outs.append((torch.full_like(q, float("nan")), torch.full((B, H, M), float("nan"), device="cuda")))
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK

    stream = torch.cuda.current_stream().cuda_stream
    free_before = torch.cuda.mem_get_info()[0]
    for (q, k, v, B, H, M, N, D, causal), (o, l) in zip(probs, outs):   # two calls in a row
        st = fa.fa_fwd_noalloc_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                                   B, H, M, N, D, 1 / math.sqrt(D), causal, stream)
        assert st == fa.FA_OK, fa.fa_last_error()
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before, "fa_fwd_noalloc changed the device's free memory"

    assert fa.fa_get_device_status() == fa.FA_OK   # reads the static array's status word too

    # Same kernel, same inputs, same schedule: the bits must be fa_fwd's.
    for (o_ref, l_ref), (o, l), case in zip(refs, outs, cases):
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref), f"noalloc differs from fa_fwd on {case}"
        check_bf16(o.float().cpu().numpy(), l.cpu().numpy(), o_ref.double().cpu().numpy(),
                   l_ref.double().cpu().numpy(), f"noalloc vs fa_fwd {case}")


def test_noalloc_rejects_what_fa_fwd_rejects(fa):
    a = 1 << 24
    assert fa.fa_fwd_noalloc_raw(a, 2 * a, 3 * a, 4 * a, 5 * a, 1, 1, 128, 128, 80, 0.1, False, 0) == \
        fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_noalloc_raw(0, 2 * a, 3 * a, 4 * a, 5 * a, 1, 1, 128, 128, 64, 0.1, False, 0) == \
        fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_noalloc_raw(a, 2 * a, 3 * a, 4 * a, 5 * a, 0, 1, 128, 128, 64, 0.1, False, 0) == fa.FA_OK

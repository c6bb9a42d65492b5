"""Back-to-back launches of every kernel family, queued without a host
synchronisation between them (the way a training or serving loop issues
them).

Each CTA's roles hand tiles to one another through mbarriers, and a wait
on a barrier is a wait for a phase parity: it is only correct while no
barrier can complete two phases before a waiter looks.  A slip in that
protocol shows up as a rare, timing-dependent wait that never ends: the
bounded wait then gives up, sets the status word and leaves the outputs
partly unwritten.  So every family here runs 40 launches over one input,
and each launch must reproduce the first launch's bits (compared on the
device, so the queue is never drained early), with a clear status word at
the end.  Sizes are the benchmark's (many persistent rounds per CTA).
"""
import pytest
import torch

pytestmark = pytest.mark.gpu
REPEATS = 40


def _inputs(B, H, N, d, seed, dtype=torch.bfloat16):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    q = torch.randn(B, N, H, d, device="cuda", dtype=dtype, generator=g)
    k = torch.randn(B, N, H, d, device="cuda", dtype=dtype, generator=g)
    v = torch.randn(B, N, H, d, device="cuda", dtype=dtype, generator=g)
    return q, k, v


def _repeat_same_bits(fa, run):
    first = [x.clone() for x in run() if x is not None]
    same = torch.ones((), dtype=torch.bool, device="cuda")
    for _ in range(REPEATS):
        out = [x for x in run() if x is not None]
        for x, y in zip(out, first):
            same &= (x == y).all()
    assert fa.fa_check_status() == fa.FA_OK
    assert bool(same.item())
    assert all(bool(torch.isfinite(x).all()) for x in first)


@pytest.mark.parametrize("d,H", [(64, 32), (128, 16), (256, 8)])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_back_to_back(gpu_lib, d, H, causal):
    fa = gpu_lib
    q, k, v = _inputs(4, H, 4096, d, seed=101)
    _repeat_same_bits(fa, lambda: fa.attention(q, k, v, causal=causal))


@pytest.mark.parametrize("window,softcap,sinks", [((1024, 0), 50.0, True), ((-1, 0), 0.0, False),
                                                  ((300, 200), 0.0, True)])
def test_forward_variants_back_to_back(gpu_lib, window, softcap, sinks):
    fa = gpu_lib
    q, k, v = _inputs(4, 16, 4096, 128, seed=102)
    s = torch.linspace(-1.0, 3.0, 16, device="cuda") if sinks else None
    _repeat_same_bits(fa, lambda: fa.attention_ext(q, k, v, window=window, softcap=softcap, sinks=s))


@pytest.mark.parametrize("causal", [False, True])
def test_packed_gqa_back_to_back(gpu_lib, causal):
    fa = gpu_lib
    g = torch.Generator(device="cuda")
    g.manual_seed(106)
    q = torch.randn(4, 4096, 16, 128, device="cuda", dtype=torch.bfloat16, generator=g)
    k = torch.randn(4, 4096, 2, 128, device="cuda", dtype=torch.bfloat16, generator=g)
    v = torch.randn(4, 4096, 2, 128, device="cuda", dtype=torch.bfloat16, generator=g)
    _repeat_same_bits(fa, lambda: fa.attention(q, k, v, causal=causal, pack_gqa=True))


def test_fp8_back_to_back(gpu_lib):
    fa = gpu_lib
    q, k, v = _inputs(4, 16, 4096, 128, seed=103)
    (q8, qs), (k8, ks), (v8, vs) = (fa.quantize_fp8(x) for x in (q, k, v))
    _repeat_same_bits(fa, lambda: fa.attention_fp8(q8, k8, v8, qs, ks, vs))


def test_splitkv_back_to_back(gpu_lib):
    fa = gpu_lib
    q, k, v = _inputs(1, 2, 16384, 128, seed=104)
    _repeat_same_bits(fa, lambda: fa.attention_splitkv(q, k, v, n_splits=4))


def test_backward_variants_back_to_back(gpu_lib):
    fa = gpu_lib
    q, k, v = _inputs(2, 16, 4096, 64, seed=105)
    do = torch.randn_like(q)
    o, lse = fa.attention_ext(q, k, v, window=(1024, 0))
    _repeat_same_bits(fa, lambda: fa.attention_backward_ext(q, k, v, o, lse, do, window=(1024, 0)))

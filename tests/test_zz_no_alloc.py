"""GPU check of fa_bwd_noalloc, the backward entry point that allocates
nothing and uses the library's own device workspace instead of one passed
by the caller (for callers that must not allocate at the point of the
call).  It runs the same kernels as fa_bwd, so its gradients must equal
fa_bwd's bit for bit.

Before the checked calls, fa_bwd_noalloc runs on a different problem
(other inputs, a larger B*H*N, the other mask), which leaves the shared
array holding values that are wrong for the checked problem: a kernel that
read the workspace before the preprocess wrote it would then differ from
fa_bwd.  Two checked calls in a row follow.  The file is named to be
collected last, so it also runs after every other test in one session.
"""
import pytest
import torch

import exact_attention_forward_fa_gb300 as fa
from exact_attention_forward_fa_gb300 import synth

pytestmark = pytest.mark.gpu


def _problem(B, H, N, d, causal, seed):
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in synth.qkv(B, H, N, d, seed=seed))
    dout = torch.from_numpy(synth.normal((B, N, H, d), seed=seed + 3)).to(q.dtype).to(dev)
    a = synth.default_alpha(d)
    o, lse = fa.attention(q, k, v, causal=causal, alpha=a)
    return q, k, v, dout, o, lse, a


def _noalloc(lib, q, k, v, o, dout, lse, B, H, N, d, a, causal):
    g = [torch.full_like(x, float("nan")) for x in (q, k, v)]
    rc = lib.fa_bwd_noalloc(q, k, v, o, dout, lse, *g, B, H, N, d, a, int(causal),
                            lib.FA_BF16)
    assert rc == lib.FA_OK
    assert lib.fa_check_status() == lib.FA_OK
    return g


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 3, 1000, 128, True), (1, 4, 777, 64, False)])
def test_noalloc_matches_fa_bwd_twice(gpu_lib, B, H, N, d, causal):
    # fill the array from another problem: 4x the rows, the other mask
    Bf, Hf, Nf = 2 * B, 2 * H, N + 129
    pf = _problem(Bf, Hf, Nf, d, not causal, seed=N + 101)
    _noalloc(gpu_lib, pf[0], pf[1], pf[2], pf[4], pf[3], pf[5], Bf, Hf, Nf, d, pf[6],
             not causal)
    q, k, v, dout, o, lse, a = _problem(B, H, N, d, causal, seed=N)
    ref = gpu_lib.attention_backward(q, k, v, o, lse, dout, causal=causal, alpha=a)
    for _ in range(2):
        g = _noalloc(gpu_lib, q, k, v, o, dout, lse, B, H, N, d, a, causal)
        for x, y in zip(g, ref):
            assert torch.equal(x, y)


def test_noalloc_limit_and_argument_codes(gpu_lib):
    lib = gpu_lib
    x = torch.zeros((1, 128, 1, 128), dtype=torch.bfloat16, device="cuda")
    l = torch.zeros((1, 1, 128), dtype=torch.float32, device="cuda")
    # 2 * B * H * 128 floats beyond 4 Mi: rejected before anything runs
    rc = lib.fa_bwd_noalloc(x, x, x, x, x, l, x, x, x, 16385, 1, 128, 128, 0.1, 0, lib.FA_BF16)
    assert rc == lib.FA_ERR_TOO_LARGE
    # an unsupported head dim gives fa_bwd's code even on a large problem
    rc = lib.fa_bwd_noalloc(x, x, x, x, x, l, x, x, x, 16385, 1, 128, 256, 0.1, 0, lib.FA_BF16)
    assert rc == lib.FA_ERR_UNSUPPORTED

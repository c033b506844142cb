"""Single-kernel parity through the per-kernel C entry points: GEMM epilogues,
prefill attention and the lm_head + argmax, each against float64 on the same
bf16 inputs."""
import numpy as np
import pytest
import torch

import oracle
from qwen3_prefill_kv_gb300 import _lib

pytestmark = pytest.mark.gpu


def _bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


def _gemm_ref(A, W, mode, N, up_off):
    a = A.double(); w = W.double()
    if mode == _lib.GEMM_SWIGLU_BF16:
        return torch.from_numpy(oracle.swiglu(torch.cat([a @ w[:N].T, a @ w[up_off:up_off + N].T], 1).numpy(), N))
    return a @ w[:N].T


GEMM_CASES = [(1, 256, 128), (37, 256, 128), (130, 384, 384), (77, 4096, 1024), (64, 1024, 2048),
              (415, 1024, 3072)]


@pytest.mark.parametrize("impl", [_lib.IMPL_SIMT, _lib.IMPL_TCGEN05], ids=["simt", "tcgen05"])
@pytest.mark.parametrize("M,N,K", GEMM_CASES)
@pytest.mark.parametrize("mode", [_lib.GEMM_STORE_F32, _lib.GEMM_ADD_F32, _lib.GEMM_SWIGLU_BF16, _lib.GEMM_STORE_BF16])
def test_gemm_epilogues(impl, M, N, K, mode):
    A = _bf16((M, K), 1)
    rows = 2 * N if mode == _lib.GEMM_SWIGLU_BF16 else N
    W = _bf16((rows, K), 2, std=0.02)
    ref = _gemm_ref(A, W, mode, N, N)
    if mode in (_lib.GEMM_STORE_F32, _lib.GEMM_ADD_F32):
        C0 = torch.randn(M, N) if mode == _lib.GEMM_ADD_F32 else torch.zeros(M, N)
        Cd = C0.cuda()
        _lib.gemm(A.cuda(), W.cuda(), M, N, K, mode, Cd, up_off=N, impl=impl)
        got = Cd.cpu().double() - (C0.double() if mode == _lib.GEMM_ADD_F32 else 0)
        tol = 2e-5 * ref.abs().max().item() + 1e-6
    else:
        Cd = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
        _lib.gemm(A.cuda(), W.cuda(), M, N, K, mode, Cd, up_off=N, impl=impl)
        got = Cd.cpu().double()
        tol = 8e-3 * ref.abs().max().item()
    torch.cuda.synchronize()
    _lib.device_error()
    assert (got - ref).abs().max().item() <= tol


WIDE_CASES = [(1, 256, 128), (130, 512, 384), (77, 4096, 1024), (300, 1024, 2048), (415, 1024, 3072)]


@pytest.mark.parametrize("tile_rows", [128, 256], ids=["128x256", "256x256"])
@pytest.mark.parametrize("M,N,K", WIDE_CASES)
@pytest.mark.parametrize("mode", [_lib.GEMM_STORE_F32, _lib.GEMM_ADD_F32, _lib.GEMM_SWIGLU_BF16, _lib.GEMM_STORE_BF16])
def test_gemm_wide_tiles(M, N, K, mode, tile_rows):
    """The tcgen05 GEMM with 256-wide tiles (SwiGLU: 128 gate + 128 up columns), forced, on
    one CTA (128 rows) and on a CTA pair (256 rows, cta_group::2: each CTA loads its own 128
    rows of A and of B; M = 1, 77, 130 and 300 leave the second CTA's rows partly or wholly
    past the end)."""
    up_off = N + 128 if mode == _lib.GEMM_SWIGLU_BF16 else 0
    rows = up_off + N if mode == _lib.GEMM_SWIGLU_BF16 else N
    A = _bf16((M, K), 21, 0.5)
    W = _bf16((rows, K), 22, 0.05)
    bf = mode in (_lib.GEMM_SWIGLU_BF16, _lib.GEMM_STORE_BF16)
    C0 = torch.zeros(M, N) if bf else _bf16((M, N), 23).float()
    Cd = C0.to(torch.bfloat16).cuda() if bf else C0.cuda()
    prev = _lib.gemm_tile_width(256)
    prev_rows = _lib.gemm_tile_rows(tile_rows)
    try:
        _lib.gemm(A.cuda(), W.cuda(), M, N, K, mode, Cd, up_off=up_off, impl=_lib.IMPL_TCGEN05)
        torch.cuda.synchronize()
    finally:
        _lib.gemm_tile_width(prev)
        _lib.gemm_tile_rows(prev_rows)
    _lib.device_error()
    ref = _gemm_ref(A, W, mode, N, up_off)
    if mode == _lib.GEMM_ADD_F32:
        ref = ref + C0.double()
    got = Cd.cpu().double()
    tol = 8e-3 if bf else 2e-5
    assert (got - ref).abs().max().item() <= tol * ref.abs().max().item() + 1e-6


def test_gemm_tile_width_rejects_other_values():
    with pytest.raises(_lib.QdecError):
        _lib.gemm_tile_width(192)
    assert _lib.gemm_tile_width(0) == 0
    with pytest.raises(_lib.QdecError):
        _lib.gemm_tile_rows(64)
    assert _lib.gemm_tile_rows(0) == 0


@pytest.mark.parametrize("M,N,K,splits", [(64, 4096, 1024, 8), (64, 1024, 3072, 32), (5, 256, 128, 2),
                                          (64, 6144, 1024, 4), (130, 1024, 2048, 3)])
def test_gemm_splitk_atomic(M, N, K, splits):
    A = _bf16((M, K), 11)
    W = _bf16((N, K), 12, std=0.02)
    C0 = torch.randn(M, N)
    Cd = C0.cuda()
    _lib.gemm_splitk(A.cuda(), W.cuda(), M, N, K, splits, Cd)
    torch.cuda.synchronize()
    _lib.device_error()
    ref = A.double() @ W.double().T
    got = Cd.cpu().double() - C0.double()
    assert (got - ref).abs().max().item() <= 2e-5 * ref.abs().max().item() + 1e-6


ATTN_CASES = [(77, 4, 2, 32, 0), (64, 16, 8, 128, 0), (200, 16, 8, 128, 0), (33, 4, 2, 32, 40), (5, 16, 8, 128, 100),
              (415, 16, 8, 128, 0), (1000, 16, 8, 128, 0), (130, 4, 4, 128, 0), (300, 8, 1, 128, 0),
              (300, 16, 8, 128, 77), (2100, 16, 8, 128, 0)]


@pytest.mark.parametrize("impl", [_lib.IMPL_SIMT, _lib.IMPL_TCGEN05], ids=["simt", "tcgen05"])
@pytest.mark.parametrize("T,HQ,HKV,D,pos0", ATTN_CASES)
def test_attention_prefill(impl, T, HQ, HKV, D, pos0):
    if impl == _lib.IMPL_TCGEN05 and D != 128:
        pytest.skip("the tensor-core attention covers head_dim 128")
    L = pos0 + T
    max_seq = L + 7
    Q = _bf16((T, HQ, D), 3)
    K = _bf16((HKV, max_seq, D), 4)
    Vv = _bf16((HKV, max_seq, D), 5)
    O = torch.zeros(T, HQ * D, dtype=torch.bfloat16, device="cuda")
    _lib.attention_prefill(Q.cuda(), T, HQ, HKV, D, max_seq, pos0, K.cuda(), Vv.cuda(), O, impl=impl)
    torch.cuda.synchronize()
    _lib.device_error()
    ref = oracle.causal_gqa_attention(Q.double().numpy(), K[:, :L].permute(1, 0, 2).double().numpy(),
                                      Vv[:, :L].permute(1, 0, 2).double().numpy(),
                                      np.arange(pos0, pos0 + T), np.arange(L)).reshape(T, HQ * D)
    got = O.cpu().double().numpy()
    assert np.abs(got - ref).max() <= 1e-2 * np.abs(ref).max()


@pytest.mark.parametrize("HQ,HKV", [(16, 8), (4, 4)])
def test_attention_prefill_rising_scores(HQ, HKV):
    """Keys whose scale grows with position make each key tile's row maximum exceed the
    running one by more than 2^8 (in the exp2 domain) every few tiles, so the tensor-core
    kernel's deferred rescaling of O is exercised; the softmax must still be exact."""
    T, D, pos0 = 1000, 128, 0
    L, max_seq = T, T
    g = torch.Generator().manual_seed(11)
    Q = (0.5 + 0.1 * torch.randn(T, HQ, D, generator=g)).to(torch.bfloat16)
    c = (torch.arange(max_seq, dtype=torch.float32) / 100.0).view(1, max_seq, 1)
    K = (c * (0.5 + 0.1 * torch.randn(HKV, max_seq, D, generator=g))).to(torch.bfloat16)
    Vv = _bf16((HKV, max_seq, D), 12)
    O = torch.zeros(T, HQ * D, dtype=torch.bfloat16, device="cuda")
    _lib.attention_prefill(Q.cuda(), T, HQ, HKV, D, max_seq, pos0, K.cuda(), Vv.cuda(), O, impl=_lib.IMPL_TCGEN05)
    torch.cuda.synchronize()
    _lib.device_error()
    ref = oracle.causal_gqa_attention(Q.double().numpy(), K.permute(1, 0, 2).double().numpy(),
                                      Vv.permute(1, 0, 2).double().numpy(), np.arange(T), np.arange(L)).reshape(T, HQ * D)
    got = O.cpu().double().numpy()
    assert np.abs(got - ref).max() <= 1e-2 * np.abs(ref).max()


@pytest.mark.parametrize("V,H", [(1024, 128), (151936, 1024), (1000, 256)])
def test_lm_head_argmax(V, H):
    E = _bf16((V, H), 6, std=0.02)
    x = torch.randn(H, generator=torch.Generator().manual_seed(7)) * 3
    g = (1 + 0.1 * torch.randn(H, generator=torch.Generator().manual_seed(8))).to(torch.bfloat16)
    scratch = torch.zeros(_lib.lm_head_scratch_bytes(V), dtype=torch.uint8, device="cuda")
    logits = torch.empty(V, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    for _ in range(2):      # the second call checks that the ticket counter was returned to zero
        _lib.lm_head_argmax(E.cuda(), V, H, x.cuda(), g.cuda(), 1e-6, logits, am, scratch)
        torch.cuda.synchronize()
        h = oracle.rms_norm(x.double().numpy(), g.double().numpy(), 1e-6)
        ref = oracle.tied_lm_head(E.double().numpy(), h)
        got = logits.cpu().double().numpy()
        assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max()
        assert int(am.item()) == int(np.argmax(got))


def test_lm_head_tie_takes_lowest_index():
    V, H = 4096, 128
    E = _bf16((V, H), 9, std=0.02)
    x = torch.randn(H, generator=torch.Generator().manual_seed(10))
    best = int(torch.argmax(E.float() @ x))
    E[3000] = E[best]; E[17] = E[best]; E[best] = E[best]      # three identical maximal rows
    g = torch.ones(H, dtype=torch.bfloat16)
    scratch = torch.zeros(_lib.lm_head_scratch_bytes(V), dtype=torch.uint8, device="cuda")
    logits = torch.empty(V, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    _lib.lm_head_argmax(E.cuda(), V, H, x.cuda(), g.cuda(), 1e-6, logits, am, scratch)
    torch.cuda.synchronize()
    assert int(am.item()) == min(17, best)

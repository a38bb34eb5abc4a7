"""Grouped (mixture-of-experts) matmul on the GPU: one launch over G experts
with per-expert rows read from a device array, on the CUDA-core (dp4a) form
and the warp-level MMA form.  Each expert's rows match the oracle (within
1e-5 per row); on dp4a they also match, bit for bit, the single-expert call
on the same rows; empty experts, an expert holding every row and experts
with more rows than a kernel's batch width (several activation tiles on the
MMA form) are covered."""
import numpy as np
import pytest
import torch

import oracle
from _gates import gate_independent, gate_parity, gate_written
from _gpu import dev, independent_fp32, oracle_matmul, oracle_q8, quantize_gpu
from iq4_xs_quantized_gb300 import binding as B
from iq4_xs_quantized_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from iq4_xs_quantized_gb300 import build
    build.build()
    B.load()
    yield
    assert B.iq4xs_last_device_error() == 0


FORMS = {B.PATH_DP4A: "dp4a", B.PATH_MMA: "mma", B.PATH_TC: "tc"}


def _run_grouped(W, rows_x, offsets, path="auto"):
    G, N, K = W.G, W.N, W.K
    w = W.weights()
    stride = w.shape[1] * w.shape[2]
    wd = dev(w.reshape(G, -1))
    qs, ds = quantize_gpu(rows_x)
    off_d = dev(offsets.astype(np.int32))
    M = rows_x.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    B.iq4xs_matmul_grouped(wd, stride, G, N, K, qs, ds, off_d, y, path=path)
    torch.cuda.synchronize()
    return w, wd, qs, ds, y.cpu().numpy()


def _check_experts(W, w, rows_x, offsets, y):
    assert gate_written(y) is None
    qs_o, d_o, _ = oracle_q8(rows_x)
    for g in range(W.G):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        if r1 > r0:
            r = gate_parity(y[r0:r1], oracle_matmul(w[g], W.N, W.K, qs_o[r0:r1], d_o[r0:r1]))
            assert r is None, (g, r)
    return qs_o, d_o


@pytest.mark.parametrize("T,topk", [(20, 4), (40, 6), (3, 2), (9, 3)])
def test_grouped_matches_oracle_and_single_expert_calls(T, topk):
    W = synth.MoEWorkload("moe_small", seed=7, G=8, N=256, K=1024, topk=topk, tokens=(T,),
                          d_scale=2e-3)
    x, rows_x, offsets = W.inputs(T)
    w, wd, qs, ds, y = _run_grouped(W, rows_x, offsets, "dp4a")
    assert gate_written(y) is None
    qs_o, d_o, _ = oracle_q8(rows_x)
    for g in range(W.G):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        if r1 == r0:
            continue
        ref = oracle_matmul(w[g], W.N, W.K, qs_o[r0:r1], d_o[r0:r1])
        r = gate_parity(y[r0:r1], ref)
        assert r is None, (g, r)
        # the single-expert call on the same rows gives the same bits
        ys = torch.full((r1 - r0, W.N), float("nan"), device="cuda")
        B.iq4xs_matmul(wd[g], W.N, W.K, qs[r0:r1], ds[r0:r1], r1 - r0, ys, B.PATH_DP4A)
        torch.cuda.synchronize()
        assert np.array_equal(ys.cpu().numpy(), y[r0:r1]), g
    ind = independent_fp32(np.concatenate([w[g] for g in range(W.G)]), W.G * W.N, W.K, qs_o, d_o)
    ind_own = np.full_like(y, np.nan)
    for g in range(W.G):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        ind_own[r0:r1] = ind[r0:r1, g * W.N:(g + 1) * W.N]
    assert gate_independent(y, ind_own) is None


@pytest.mark.parametrize("T,topk", [(20, 4), (40, 6), (9, 3), (64, 8)])
def test_grouped_mma_matches_oracle(T, topk):
    """The warp-MMA form over larger per-expert batches (ragged N)."""
    W = synth.MoEWorkload("moe_mma", seed=17, G=8, N=200, K=1024, topk=topk, tokens=(T,),
                          d_scale=2e-3)
    _, rows_x, offsets = W.inputs(T)
    w, wd, qs, ds, y = _run_grouped(W, rows_x, offsets, "mma")
    qs_o, d_o = _check_experts(W, w, rows_x, offsets, y)
    ind = independent_fp32(np.concatenate([w[g] for g in range(W.G)]), W.G * W.N, W.K, qs_o, d_o)
    ind_own = np.full_like(y, np.nan)
    for g in range(W.G):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        ind_own[r0:r1] = ind[r0:r1, g * W.N:(g + 1) * W.N]
    assert gate_independent(y, ind_own) is None
    # AUTO takes the form the host query names (its rule is pinned on the
    # CPU); same bits as the explicit call
    M = rows_x.shape[0]
    auto = FORMS[B.iq4xs_select_grouped_path(W.G, W.N, W.K, M)]
    y_auto = _run_grouped(W, rows_x, offsets)[-1]
    y_expl = y if auto == "mma" else _run_grouped(W, rows_x, offsets, auto)[-1]
    assert np.array_equal(y_auto, y_expl), auto


@pytest.mark.parametrize("T,topk,G", [(64, 8, 8), (256, 8, 16), (1024, 4, 8), (40, 6, 8)])
def test_grouped_tc_matches_oracle(T, topk, G):
    """The tcgen05 form over per-expert batches from a few rows to several
    128-row tiles (ragged N; tiles of the layer mapped to experts in-kernel),
    against the oracle and an independent fp32 product."""
    W = synth.MoEWorkload("moe_tc", seed=23, G=G, N=200, K=1024, topk=topk, tokens=(T,), d_scale=2e-3)
    _, rows_x, offsets = W.inputs(T)
    w, wd, qs, ds, y = _run_grouped(W, rows_x, offsets, "tc")
    qs_o, d_o = _check_experts(W, w, rows_x, offsets, y)
    ind = independent_fp32(np.concatenate([w[g] for g in range(W.G)]), W.G * W.N, W.K, qs_o, d_o)
    ind_own = np.full_like(y, np.nan)
    for g in range(W.G):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        ind_own[r0:r1] = ind[r0:r1, g * W.N:(g + 1) * W.N]
    assert gate_independent(y, ind_own) is None
    # AUTO takes the tcgen05 form from 32 mean rows per expert slot on
    M = rows_x.shape[0]
    if B.iq4xs_select_grouped_path(W.G, W.N, W.K, M) == B.PATH_TC:
        assert np.array_equal(_run_grouped(W, rows_x, offsets)[-1], y)


@pytest.mark.parametrize("path", ("dp4a", "mma", "tc"))
@pytest.mark.parametrize("G,T,topk", [(70, 5, 2), (100, 40, 3)])
def test_grouped_many_experts_compacted_slots(G, T, topk, path):
    # more experts than a warp's ballot covers; fewer (and more) rows than experts
    W = synth.MoEWorkload("moe_wide", seed=13, G=G, N=128, K=512, topk=topk, tokens=(T,),
                          d_scale=2e-3)
    _, rows_x, offsets = W.inputs(T)
    w, wd, qs, ds, y = _run_grouped(W, rows_x, offsets, path)
    _check_experts(W, w, rows_x, offsets, y)


@pytest.mark.parametrize("path", ("dp4a", "mma", "tc"))
@pytest.mark.parametrize("rows", (11, 80, 300))
def test_grouped_empty_experts_and_one_expert_with_every_row(path, rows):
    """80 rows on one expert: five activation tiles of 16 rows in one CTA on
    the MMA form (the tile from the mean rows of the six expert slots)."""
    W = synth.MoEWorkload("moe_edge", seed=9, G=6, N=128, K=512, topk=1, tokens=(rows,),
                          d_scale=2e-3)
    rng = np.random.default_rng(11)
    rows_x = synth.activations(rng, rows, W.K)
    offsets = np.array([0, 0, 0, rows, rows, rows, rows], dtype=np.int32)  # all rows on expert 2
    w, wd, qs, ds, y = _run_grouped(W, rows_x, offsets, path)
    assert gate_written(y) is None
    qs_o, d_o, _ = oracle_q8(rows_x)
    assert gate_parity(y, oracle_matmul(w[2], W.N, W.K, qs_o, d_o)) is None


@pytest.mark.parametrize("path", ("dp4a", "mma", "tc"))
def test_grouped_padded_expert_stride_and_ldy(path):
    """Experts 512 bytes apart beyond their matrices and y rows wider than N:
    every form reads only its expert's rows and writes only columns < N."""
    W = synth.MoEWorkload("moe_pad", seed=29, G=5, N=136, K=1024, topk=2, tokens=(150,), d_scale=2e-3)
    _, rows_x, offsets = W.inputs(150)
    w = W.weights()
    G, N, K = W.G, W.N, W.K
    mat = w.shape[1] * w.shape[2]
    stride = mat + 512
    buf = np.full((G, stride), 0xA5, dtype=np.uint8)  # the padding holds garbage blocks
    buf[:, :mat] = w.reshape(G, -1)
    qs, ds = quantize_gpu(rows_x)
    M, ldy = rows_x.shape[0], N + 7
    y = torch.full((M, ldy), float("nan"), dtype=torch.float32, device="cuda")
    B.iq4xs_matmul_grouped(dev(buf), stride, G, N, K, qs, ds, dev(offsets.astype(np.int32)), y, path=path)
    torch.cuda.synchronize()
    yn = y.cpu().numpy()
    assert np.all(np.isnan(yn[:, N:])), "columns beyond N must not be written"
    _check_experts(W, w, rows_x, offsets, np.ascontiguousarray(yn[:, :N]))


def test_grouped_rejects_bad_arguments():
    W = synth.MoEWorkload("moe_arg", seed=1, G=2, N=128, K=512, topk=1, tokens=(2,), d_scale=2e-3)
    w = dev(W.weights().reshape(2, -1))
    qs, ds = B.alloc_activations(2, W.K, "cuda")
    off = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    y = torch.empty((2, W.N), device="cuda")
    stride = w.shape[1]
    with pytest.raises(B.IQ4XSError) as e:
        B.iq4xs_matmul_grouped(w, stride - 16, 2, W.N, W.K, qs, ds, off, y)
    assert e.value.status == B.ERR_ARG
    with pytest.raises(B.IQ4XSError) as e:
        B.iq4xs_matmul_grouped(w, stride, 0, W.N, W.K, qs, ds, off, y)
    assert e.value.status == B.ERR_SHAPE
    with pytest.raises(B.IQ4XSError) as e:
        B.iq4xs_matmul_grouped(w, stride, 2, W.N, W.K, qs, ds, off, y, path=B.PATH_BASELINE)
    assert e.value.status == B.ERR_ARG
    W3 = synth.MoEWorkload("moe_k768", seed=1, G=2, N=128, K=768, topk=1, tokens=(2,), d_scale=2e-3)
    w3 = dev(W3.weights().reshape(2, -1))
    qs3, ds3 = B.alloc_activations(2, 768, "cuda")
    for p in ("mma", "tc"):  # the tensor-core forms need K % 512 == 0
        with pytest.raises(B.IQ4XSError) as e:
            B.iq4xs_matmul_grouped(w3, w3.shape[1], 2, W3.N, 768, qs3, ds3, off, y, path=p)
        assert e.value.status == B.ERR_SHAPE


@pytest.mark.parametrize("wt", (B.WTYPE_Q4_0, B.WTYPE_IQ4_NL))
@pytest.mark.parametrize("path", ("dp4a", "mma", "auto"))
@pytest.mark.parametrize("T,topk,G", [(20, 4, 8), (3, 2, 70), (64, 8, 16)])
def test_grouped_formats_match_oracle(wt, path, T, topk, G):
    """Q4_0 / IQ4_NL experts on the CUDA-core and persistent warp-MMA forms
    (and AUTO, which keeps them off the tcgen05 form): every expert's rows
    against the oracle's matmul of that format, and bitwise against
    iq4xs_matmul_wt on the same path over the expert's rows."""
    W = synth.MoEWorkload("moe_formats", seed=31, G=G, N=200, K=1024, topk=topk, tokens=(T,), d_scale=2e-3)
    _, rows_x, offsets = W.inputs(T)
    N, K = W.N, W.K
    w = np.stack([synth.block32_weights(np.random.default_rng([31, wt, g]), N, K, 2e-3) for g in range(G)])
    stride = w.shape[1] * w.shape[2]
    wd = dev(w.reshape(G, -1))
    qs, ds = quantize_gpu(rows_x)
    off_d = dev(offsets.astype(np.int32))
    M = rows_x.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    B.iq4xs_matmul_grouped(wd, stride, G, N, K, qs, ds, off_d, y, path=path, wtype=wt)
    torch.cuda.synchronize()
    yn = y.cpu().numpy()
    assert gate_written(yn) is None
    qs_o, d_o, _ = oracle_q8(rows_x)
    orc = oracle.get()
    form = path if path != "auto" else FORMS[B.iq4xs_select_grouped_path(G, N, K, M, wt)]
    assert form != "tc"
    for g in range(G):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        if r1 > r0:
            r = gate_parity(yn[r0:r1], orc.matmul_wt(wt, w[g], N, K, qs_o[r0:r1], d_o[r0:r1]))
            assert r is None, (g, r)
            if form == "dp4a":  # the CUDA-core form: each expert with its own batch width
                ys = torch.full((r1 - r0, N), float("nan"), dtype=torch.float32, device="cuda")
                B.iq4xs_matmul_wt(wd[g], wt, N, K, qs[r0:r1], ds[r0:r1], r1 - r0, ys, B.PATH_DP4A)
                torch.cuda.synchronize()
                assert np.array_equal(ys.cpu().numpy(), yn[r0:r1]), g


def test_grouped_formats_reject_the_tcgen05_form():
    G, N, K = 4, 128, 512
    w = torch.zeros((G, N * (K // 32) * 18), dtype=torch.uint8, device="cuda")
    qs, ds = B.alloc_activations(8, K, "cuda")
    off = torch.tensor([0, 2, 4, 6, 8], dtype=torch.int32, device="cuda")
    y = torch.empty((8, N), device="cuda")
    with pytest.raises(B.IQ4XSError) as e:
        B.iq4xs_matmul_grouped(w, w.shape[1], G, N, K, qs, ds, off, y, path="tc", wtype=B.WTYPE_Q4_0)
    assert e.value.status == B.ERR_SHAPE

"""Dense few-row projections on the GPU (QPN2 NVFP4, QPN8 channel-FP8) and the
load-time helpers of their formats, against the oracle.

  * the channel-FP8 quantiser and the prepared-scale expansion are bit-exact
    (both layouts; the fragment layout undone from its header definition);
  * projections: rel-L2 <= 1e-3 and max-abs <= 2e-2 against the FP64-summed
    oracle on the same quantised weights;
  * batch invariance, bitwise: M = 9 / 15 / 16 / 17 / 24 / 31 / 32 equal the
    concatenated M = 8 calls ("[SM70][Draft] Extend Qwen3.8 DFlash2
    concurrency paths", sections "TP4-only NVFP4 verifier follow-up" and
    "Follow-up: exact channel-FP8 QPN8 concurrency paths");
  * prepared FP16 scales give bitwise the raw-scale output ("[Kernel][SM70]
    Improve Qwen3.8 no-MTP concurrency", section "Test Result").
"""
import numpy as np
import pytest
import torch

import oracle
from harness import MAX_ABS_TOL, REL_L2_TOL, compare
from nvfp4_weight_mixture_gb300 import moe, synth

pytestmark = pytest.mark.gpu

GU = synth.DENSE_WORKLOADS["dense_gate_up_m16"]
DN = synth.DENSE_WORKLOADS["dense_down_m16"]
SMALL = synth.DENSE_WORKLOADS["dense_small"]


def fp8_fragment_to_canonical(qf, rows, k):
    """Undo MOE_LAYOUT_FP8_FRAGMENT (header definition): block (G, ks, j) of
    1024 bytes; lane L = 4g + c holds row 16 rt + g at [16L, 16L + 16) and row
    16 rt + g + 8 at [512 + 16L, ...), elements [64 ks + 16 c, + 16)."""
    b = qf.reshape(rows // 256, k // 64, 16, 2, 8, 4, 16)   # G, ks, j, half, g, c, e
    # -> rows: G, j, half, g ; cols: ks, c, e
    return b.transpose(0, 2, 3, 4, 1, 5, 6).reshape(rows, k)


class _Dense:
    """One dense weight matrix quantised both ways (GPU fragment layouts for the
    kernels, canonical by the oracle for the reference)."""

    def __init__(self, wl):
        self.wl = wl
        w = synth.dense_weight(wl)
        wt = torch.from_numpy(w).cuda()
        self.nv = moe.quantize(wt[None], moe.LAYOUT_FRAGMENT)
        self.nv = (self.nv[0].reshape(-1), self.nv[1].reshape(-1), self.nv[2])
        self.nv_prep = (self.nv[0], moe.prepare_scales(self.nv[1]), self.nv[2])
        self.f8q, self.f8cs = moe.fp8_quantize(wt, moe.LAYOUT_FP8_FRAGMENT)
        q, s, g, st = oracle.quantize(w[None])
        assert st == 0
        self.o_nv = (q[0], s[0], float(g[0]))
        self.o_f8 = oracle.fp8_quantize(w)[:2]

    def x(self, M, variant=0):
        wl = synth.dense_with_tokens(self.wl, M)
        return synth.dense_activations(wl, variant)

    def gpu(self, fmt, x, ws=None):
        xt = torch.from_numpy(x).cuda()
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fmt == "nvfp4":
            y = moe.dense(xt, self.nv, self.wl.N, status=st, ws=ws)
        elif fmt == "prepared":
            y = moe.dense(xt, self.nv_prep, self.wl.N, prepared=True, status=st, ws=ws)
        else:
            y = moe.fp8_dense(xt, self.f8q, self.f8cs, status=st, ws=ws)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        return y.cpu().numpy()

    def ref(self, fmt, x):
        if fmt == "fp8":
            return oracle.fp8_dense(x, *self.o_f8)
        q, s, g = self.o_nv
        return oracle.dense(x, q, s, g)


_mats = {}


def _mat(wl):
    if wl.name not in _mats:
        _mats[wl.name] = _Dense(wl)
    return _mats[wl.name]


# ---- load-time helpers: bit-exact ------------------------------------------------------

def test_fp8_quantize_bit_exact_both_layouts():
    rng = np.random.default_rng(31)
    rows, k = 512, 4352
    w = (rng.standard_normal((rows, k)) * 0.02).astype(np.float32)
    w[7] = 0.0
    w[9, :5] = [3e4, -1e-9, 2e-7, 448.0, -0.0]
    w[11, 100] = np.nan
    q_ref, cs_ref, st_ref = oracle.fp8_quantize(w)
    wt = torch.from_numpy(w).cuda()
    for layout in (moe.LAYOUT_CANONICAL, moe.LAYOUT_FP8_FRAGMENT):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        q, cs = moe.fp8_quantize(wt, layout, status=st)
        torch.cuda.synchronize()
        q = q.cpu().numpy()
        if layout == moe.LAYOUT_FP8_FRAGMENT:
            q = fp8_fragment_to_canonical(q, rows, k)
        np.testing.assert_array_equal(q.reshape(rows, k), q_ref)
        np.testing.assert_array_equal(cs.cpu().numpy(), cs_ref)
        assert int(st.item()) == st_ref == oracle.ST_NONFINITE


@pytest.mark.parametrize("n", [256 * 16, 256 * 16 + 5])
def test_prepare_scales_bit_exact(n):
    codes = (np.arange(n) * 37 % 256).astype(np.uint8)       # every code, and a ragged tail
    ref, st_ref = oracle.prepare_scales(codes)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = moe.prepare_scales(torch.from_numpy(codes).cuda(), status=st)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint16), ref)
    assert int(st.item()) == st_ref == oracle.ST_NONFINITE


# ---- projections vs the oracle -----------------------------------------------------------

@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
@pytest.mark.parametrize("wl,M", [(SMALL, 1), (SMALL, 8), (SMALL, 13), (GU, 16), (GU, 32),
                                  (DN, 1), (DN, 16), (DN, 27)])
def test_dense_vs_oracle(fmt, wl, M):
    d = _mat(wl)
    x = d.x(M)
    rel, mx = compare(d.gpu(fmt, x), d.ref(fmt, x))
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (rel, mx)


# ---- batch invariance: rows equal to the same rows of concatenated M = 8 calls --------------

@pytest.mark.parametrize("fmt", ["nvfp4", "fp8", "prepared"])
@pytest.mark.parametrize("wl", [GU, DN], ids=["gate_up", "down"])
def test_dense_batch_invariance(fmt, wl):
    d = _mat(wl)
    x32 = d.x(32, variant=3)
    parts = np.concatenate([d.gpu(fmt, x32[i:i + 8]) for i in range(0, 32, 8)])
    for M in (9, 15, 16, 17, 24, 31, 32):
        y = d.gpu(fmt, np.ascontiguousarray(x32[:M]))
        np.testing.assert_array_equal(y.view(np.uint16), parts[:M].view(np.uint16), err_msg=str(M))
    # and single rows
    y1 = d.gpu(fmt, np.ascontiguousarray(x32[5:6]))
    np.testing.assert_array_equal(y1.view(np.uint16), parts[5:6].view(np.uint16))


# Shapes the layer workloads do not reach: one 256-row group (16 blocks of one
# tile), K of 5 and 17 segments (stages only partly used), and 1024 tiles over
# the 152 blocks (6 or 7 each: more than one group of 4 tiles in hand).
ODD = [synth.DenseWorkload("dense_one_group", 53, 8, 256, 320),
       synth.DenseWorkload("dense_many_tiles", 54, 8, 16384, 1088)]


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8", "prepared"])
@pytest.mark.parametrize("wl", ODD, ids=[w.name for w in ODD])
def test_dense_other_shapes_vs_oracle_and_batch(fmt, wl):
    d = _mat(wl)
    x = d.x(20, variant=2)
    y = d.gpu(fmt, x)
    rel, mx = compare(y, d.ref("fp8" if fmt == "fp8" else "nvfp4", x))
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (rel, mx)
    # rows equal to the same rows of smaller calls (M 20 against 8 + 12)
    a = d.gpu(fmt, np.ascontiguousarray(x[:8]))
    b = d.gpu(fmt, np.ascontiguousarray(x[8:]))
    np.testing.assert_array_equal(y.view(np.uint16), np.concatenate([a, b]).view(np.uint16))


@pytest.mark.parametrize("wl,M", [(GU, 1), (GU, 16), (DN, 8), (DN, 32), (SMALL, 3)])
def test_dense_prepared_scales_bitwise_equal_raw(wl, M):
    d = _mat(wl)
    x = d.x(M, variant=1)
    np.testing.assert_array_equal(d.gpu("prepared", x).view(np.uint16),
                                  d.gpu("nvfp4", x).view(np.uint16))


def test_dense_edges():
    d = _mat(SMALL)
    # M = 0: nothing to do
    x0 = torch.empty((0, SMALL.K), dtype=torch.float16, device="cuda")
    assert moe.dense(x0, d.nv, SMALL.N).shape == (0, SMALL.N)
    # M above the weight-streaming path is refused
    x33 = torch.zeros((33, SMALL.K), dtype=torch.float16, device="cuda")
    with pytest.raises(moe.MoEError):
        moe.dense(x33, d.nv, SMALL.N)
    # no output is split between blocks: no workspace, and NULL is accepted
    g = _mat(GU)
    assert moe.dense_query(16, GU.N, GU.K) == 0
    x = torch.from_numpy(g.x(16)).cuda()
    y0 = moe.dense(x, g.nv, GU.N, ws=None)
    # repeated calls are bitwise equal
    a = g.gpu("nvfp4", g.x(16))
    b = g.gpu("nvfp4", g.x(16))
    np.testing.assert_array_equal(a.view(np.uint16), b.view(np.uint16))
    np.testing.assert_array_equal(y0.cpu().numpy().view(np.uint16), a.view(np.uint16))


def test_dense_graph_replay_changing_inputs():
    d = _mat(DN)
    xs = torch.from_numpy(d.x(16)).cuda()
    ws = torch.zeros(max(moe.dense_query(16, DN.N, DN.K), 16), dtype=torch.uint8, device="cuda")
    y = torch.empty((16, DN.N), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe.fp8_dense(xs, d.f8q, d.f8cs, y=y, ws=ws)
    torch.cuda.current_stream().wait_stream(s)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        moe.fp8_dense(xs, d.f8q, d.f8cs, y=y, ws=ws)
    for v in (4, 5):
        xv = d.x(16, variant=v)
        xs.copy_(torch.from_numpy(xv).cuda())
        y.fill_(float("nan"))
        gr.replay()
        torch.cuda.synchronize()
        rel, mx = compare(y.cpu().numpy(), d.ref("fp8", xv))
        assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (v, rel, mx)

"""GPU-vs-oracle harness: one seeded layer instance on both sides.

Inputs come from ``synth`` only.  The CUDA side quantises the FP32 weights
with ``moe_nvfp4_quantize`` into the fragment layouts; the oracle quantises the
same FP32 weights itself (canonical layout) for the experts it needs.  No
value computed by the CUDA path is ever passed to the oracle.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
from nvfp4_weight_mixture_gb300 import moe, synth

_POOL = ThreadPoolExecutor(8)

REL_L2_TOL = 1e-3      # layer output vs the FP32-accumulated oracle
MAX_ABS_TOL = 2e-2
ROUTER_GAP = 1e-5      # top-k sets must agree unless the k-th / k+1-th gap is below this
ROUTER_W_TOL = 1e-5


def compare(y, yref):
    a = np.asarray(y, np.float64)
    b = np.asarray(yref, np.float64)
    den = np.linalg.norm(b.ravel())
    rel = float(np.linalg.norm((a - b).ravel()) / (den if den > 0 else 1.0))
    mx = float(np.max(np.abs(a - b))) if a.size else 0.0
    return rel, mx


def gen(fn, wl, experts):
    return list(_POOL.map(lambda e: fn(wl, e), experts))


class Case:
    """One layer: seeded inputs, GPU-quantised weights, lazily built oracle weights."""

    def __init__(self, wl, variant=0, chunk=32):
        self.wl = wl
        self.x = synth.activations(wl, variant)
        self.wr = synth.router_weight(wl)
        self.bias = synth.router_bias(wl)
        self.wg = synth.gate_weight(wl)
        dev = torch.device("cuda")
        E, H, I = wl.E, wl.H, wl.I
        self.q13 = torch.empty((E, I * H), dtype=torch.uint8, device=dev)
        self.s13 = torch.empty((E, I * H // 8), dtype=torch.uint8, device=dev)
        self.g13 = torch.empty((E,), dtype=torch.float32, device=dev)
        self.q2 = torch.empty((E, H * I // 2), dtype=torch.uint8, device=dev)
        self.s2 = torch.empty((E, H * I // 16), dtype=torch.uint8, device=dev)
        self.g2 = torch.empty((E,), dtype=torch.float32, device=dev)
        for e0 in range(0, E, chunk):
            e1 = min(E, e0 + chunk)
            w = torch.from_numpy(np.stack(gen(synth.expert_w13, wl, range(e0, e1)))).to(dev)
            moe.quantize(w, moe.LAYOUT_FRAGMENT_W13, q=self.q13[e0:e1], s=self.s13[e0:e1],
                         g=self.g13[e0:e1])
            w = torch.from_numpy(np.stack(gen(synth.expert_w2, wl, range(e0, e1)))).to(dev)
            moe.quantize(w, moe.LAYOUT_FRAGMENT, q=self.q2[e0:e1], s=self.s2[e0:e1],
                         g=self.g2[e0:e1])
        self.sh13 = self.sh2 = None
        if wl.shared:
            self.sh13 = moe.quantize(torch.from_numpy(synth.shared_w13(wl)).to(dev),
                                     moe.LAYOUT_FRAGMENT_W13)
            self.sh2 = moe.quantize(torch.from_numpy(synth.shared_w2(wl)).to(dev),
                                    moe.LAYOUT_FRAGMENT)
        self.x_t = torch.from_numpy(self.x).to(dev)
        self.layer = moe.MoELayer(
            H, E, wl.k, I, torch.from_numpy(self.wr).to(dev), (self.q13, self.s13, self.g13),
            (self.q2, self.s2, self.g2), self.sh13, self.sh2,
            None if self.wg is None else torch.from_numpy(self.wg).to(dev),
            None if self.bias is None else torch.from_numpy(self.bias).to(dev),
            max_tokens=max(wl.M, 1))
        self._o13 = None
        self._have = set()
        self._oshared = None

    # ---- oracle side ---------------------------------------------------------------
    def oracle_weights(self, experts=None):
        wl = self.wl
        E, H, I = wl.E, wl.H, wl.I
        if self._o13 is None:
            self._o13 = (np.zeros((E, 2 * I, H // 2), np.uint8), np.zeros((E, 2 * I, H // 16), np.uint8),
                         np.ones((E,), np.float32))
            self._o2 = (np.zeros((E, H, I // 2), np.uint8), np.zeros((E, H, I // 16), np.uint8),
                        np.ones((E,), np.float32))
        need = sorted(set(range(E) if experts is None else experts) - self._have)
        if need:
            def one(e):
                q, s, g, st = oracle.quantize(synth.expert_w13(wl, e)[None])
                q2, s2, g2, st2 = oracle.quantize(synth.expert_w2(wl, e)[None])
                return e, (q[0], s[0], g[0]), (q2[0], s2[0], g2[0])
            for e, a, b in _POOL.map(one, need):
                for i in range(3):
                    self._o13[i][e] = a[i]
                    self._o2[i][e] = b[i]
            self._have.update(need)
        if wl.shared and self._oshared is None:
            a = oracle.quantize(synth.shared_w13(wl)[None])
            b = oracle.quantize(synth.shared_w2(wl)[None])
            self._oshared = ((a[0][0], a[1][0], a[2][0]), (b[0][0], b[1][0], b[2][0]))
        return self._o13, self._o2, self._oshared

    def oracle_route(self, tokens=None):
        """Oracle router on the given tokens (all by default): (logits, ids, w, gamma)."""
        x = self.x if tokens is None else self.x[np.asarray(tokens)]
        logits, ids, w = oracle.router(x, self.wr, self.bias, self.wl.k)
        gamma = oracle.shared_gate(x, self.wg) if self.wl.shared else None
        return logits, ids, w, gamma

    def oracle_forward(self, tokens=None, ids=None, w=None):
        """Oracle layer output for `tokens` (all by default), routed by the oracle
        router unless ids / w (full [M, k] arrays) are given."""
        wl = self.wl
        tok = np.arange(wl.M) if tokens is None else np.asarray(tokens)
        if ids is None:
            _, ids_t, w_t, _ = self.oracle_route(tok)
            ids = np.zeros((wl.M, wl.k), np.int32)
            w = np.zeros((wl.M, wl.k), np.float32)
            ids[tok] = ids_t
            w[tok] = w_t
        gamma = None
        if wl.shared:
            gamma = np.zeros((wl.M,), np.float32)
            gamma[tok] = oracle.shared_gate(self.x[tok], self.wg)
        used = set(int(e) for e in np.asarray(ids)[tok].ravel() if 0 <= e < wl.E)
        o13, o2, osh = self.oracle_weights(used)
        y, st = oracle.forward(self.x, ids, w, o13, o2, shared=osh, gamma=gamma,
                               tokens=None if tokens is None else tok)
        return y

    # ---- GPU side ------------------------------------------------------------------
    def gpu_route(self):
        ids, w = self.layer.route(self.x_t)
        return ids.cpu().numpy(), w.cpu().numpy()

    def gpu_forward(self, ids=None, w=None, ids_from_oracle=False):
        """GPU plan + forward.  ids/w (numpy) are planned as given; with
        ids_from_oracle the oracle router's choice for all tokens is given."""
        if ids_from_oracle:
            _, ids, w, _ = self.oracle_route()
        if ids is not None:
            self.layer.route(self.x_t, torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda(),
                             torch.from_numpy(np.ascontiguousarray(w, np.float32)).cuda())
        else:
            self.layer.route(self.x_t)
        y = self.layer.forward_planned(self.x_t)
        torch.cuda.synchronize()
        return y.cpu().numpy()

    def plan_arrays(self):
        """The plan buffer decoded on the host (for bit-exact plan tests)."""
        return decode_plan(self.layer.plan_buf, self.wl.M, self.wl.k + int(self.wl.shared),
                           self.wl.E + int(self.wl.shared), self.wl.E, self.wl.H)


TILE_ROWS = 192
PLAN_CHUNK = 2048
DECODE_MAX_TOKENS = 16
DTAB_INTS = 20
DTAB_ENTRIES = DECODE_MAX_TOKENS * 33


def _align(v, a=256):
    return (v + a - 1) // a * a


def decode_plan(buf, M, k_eff, e_eff, E, H):
    """Reads the plan arrays out of the plan buffer.  The carving (256-byte
    aligned arrays in a fixed order) is the library's private layout; it is
    restated here only so that the tests can compare the plan bit for bit."""
    b = buf.cpu().numpy()
    off = 0
    P = M * k_eff
    Pc = max(P, 1)
    max_tiles = e_eff + (P + TILE_ROWS - 1) // TILE_ROWS

    def take(nbytes, dtype, count):
        nonlocal off
        a = b[off:off + count * np.dtype(dtype).itemsize].view(dtype)
        off = _align(off + nbytes)
        return a

    hdr = take(64, np.int32, 16)
    take(256, np.uint32, 64)
    ids = take(4 * Pc, np.int32, P)
    w = take(4 * Pc, np.float32, P)
    counts = take(4 * e_eff, np.int32, e_eff)
    offsets = take(4 * (e_eff + 1), np.int32, e_eff + 1)
    active = take(4 * e_eff, np.int32, e_eff)
    perm = take(4 * Pc, np.int32, P)
    inv = take(4 * Pc, np.int32, P)
    tiles = take(16 * max_tiles, np.int32, 4 * max_tiles).reshape(-1, 4)
    n_chunks = (Pc + PLAN_CHUNK - 1) // PLAN_CHUNK
    take(4 * n_chunks * e_eff, np.int32, 0)                      # chunk histograms
    take(4 * Pc, np.int32, 0)                                     # ranks
    take(4 * ((H + 127) // 128) * DECODE_MAX_TOKENS * E, np.float32, 0)  # router partials
    take(4 * DECODE_MAX_TOKENS * E, np.float32, 0)                # router logits
    dtab = take(4 * DTAB_ENTRIES * DTAB_INTS, np.int32,
                DTAB_ENTRIES * DTAB_INTS).reshape(DTAB_ENTRIES, DTAB_INTS)
    n_valid, n_active, n_tiles = int(hdr[5]), int(hdr[3]), int(hdr[4])
    return dict(hdr=hdr, ids=ids, w=w, counts=counts, offsets=offsets,
                active=active[:n_active], perm=perm[:n_valid], inv=inv,
                tiles=tiles[:n_tiles, :3], tile_pos=tiles[:n_tiles, 3], dtab=dtab)


def expected_tile_pos(ref):
    """The first plan position of each tile of an oracle plan: its expert's
    offset plus the tile's first row (the fourth field of a tile entry)."""
    t = np.asarray(ref["tiles"]).reshape(-1, 3)
    return (np.asarray(ref["offsets"])[t[:, 0]] + t[:, 1]).astype(np.int32)


def expected_work_table(ref, M, k_eff, e_eff):
    """The decode work table an oracle plan implies (M <= 16): one entry per
    active expert in ascending order, (expert, first plan position, rows, -1,
    the pair ids of its first 16 rows, -1 past them); entries from n_active to
    min(M * k_eff, e_eff) all -1.  Restated from the table's definition."""
    P = M * k_eff
    max_active = min(P, e_eff)
    out = np.full((max_active, DTAB_INTS), -1, np.int32)
    active = np.nonzero(ref["counts"])[0]
    for a, e in enumerate(active):
        off, cnt = int(ref["offsets"][e]), int(ref["counts"][e])
        out[a, 0], out[a, 1], out[a, 2] = e, off, cnt
        n = min(cnt, DTAB_INTS - 4)
        out[a, 4:4 + n] = ref["perm"][off:off + n]
    return out

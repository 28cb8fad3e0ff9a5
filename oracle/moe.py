"""Oracle: the routed-expert MoE layer, step by step, on the CPU (plain numpy, slow on purpose).

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may
import this module; the product path never does, and nothing here is shared with the CUDA code.

The pages ("New Deepseek 4.1 flash recipe" forum thread; the spark-ds41f README; the TP4 serving
profile README) describe the layer only in words. The steps and the readings taken where they
are silent:

1. Router (post 6 "How it works" item 3: TileKernels' MoE top-k gate; the "Kernel by kernel"
   table's Router row). logit[t, e] = x[t] . Wr[e] in fp32 in one FIXED order (post 6 "Why
   TileLang": every kernel adds its reductions in a fixed order): h is cut into consecutive
   chunks of 64; each chunk is accumulated sequentially from +0 in fp32; the chunk sums are then
   added left to right from +0. bf16 x bf16 products are exact in fp32, so a fused multiply-add
   and a multiply followed by an add give the same bits.
   score = sigmoid(logit) computed from IEEE fp32 +, -, *, / only (self-written exp: Cody-Waite
   reduction by ln 2 followed by the degree-7 Taylor polynomial in Horner form, then an exact
   scaling by 2^n), so that both sides of a comparison can reproduce it bit for bit.
   key = score + bias[e] (the bias only selects). Top-k by key descending, exact ties to the
   LOWER expert index (post 4, "Exact indexer selections": ties break by lowest position).
   weights w_j = score_j / ((score_0 + score_1) + ...), summed in rank order, fp32.
2. Dead rows (post 2, "Speculative decoding": dead verification rows skip the MoE expert weight
   reads): a dead row is still routed, takes no slot, and its output row is +0.0.
3. Plan: live slots grouped by expert; inside an expert ordered by token index t.
4. MXFP8 quantisation of x per 32-block (formats.scale_exponent / encode_e4m3).
5. W13: g = Wg x^, u = Wu x^ exactly (float64, all operands exact decoded values);
   a = silu(g) * u = g * sigmoid(g) * u in float64. Requantisation of a to MXFP8 per 32 along I
   takes its decisions in fp32, the precision of the kernel's epilogue: a is first rounded to
   fp32 (TileKernels "quantization with fused SwiGLU", post 6 "Why TileLang" list).
6. W2 per slot: y = w_slot * (W2 h^) in float64.
7. Combine (TP4 profile README, settings table, "Experts" row: a per-slot buffer and a
   fixed-order sum instead of atomics): out[t] = bf16_rne(((y_0 + y_1) + y_2) + ...), j in rank
   order, in float64, rounded once.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import formats as F

ROUTER_CHUNK = 64
SIGMOID_CLAMP = np.float32(80.0)

# Constants of the self-written exp, all derived from the mathematics in plain float64 and then
# rounded once to fp32. LN2_HI keeps 16 significant bits, so n * LN2_HI is exact for |n| < 2^8.
_LN2 = np.log(2.0)
LOG2E_F = np.float32(1.0 / _LN2)
LN2_HI_F = np.float32(np.round(_LN2 * 65536.0) / 65536.0)
LN2_LO_F = np.float32(_LN2 - float(LN2_HI_F))
# 1/k! for k = 7 .. 0 (Horner order)
_INV_FACT = [np.float32(1.0 / np.prod(np.arange(1, k + 1, dtype=np.float64))) for k in range(7, -1, -1)]


def exp_f32(t: np.ndarray) -> np.ndarray:
    """exp(t) for fp32 t in [-80, 80], from fp32 +, -, * only (each op rounded to nearest even)."""
    t = np.asarray(t, dtype=np.float32)
    n = np.rint(t * LOG2E_F).astype(np.float32)            # nearest integer, ties to even
    r = (t - n * LN2_HI_F).astype(np.float32)              # n*LN2_HI exact; difference exact
    r = (r - n * LN2_LO_F).astype(np.float32)
    p = np.full_like(r, _INV_FACT[0])
    for c in _INV_FACT[1:]:
        p = (p * r).astype(np.float32)
        p = (p + c).astype(np.float32)
    two_n = ((n.astype(np.int32) + 127) << 23).astype(np.int32).view(np.float32)
    return (p * two_n).astype(np.float32)


def sigmoid_f32(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float32)
    t = np.minimum(np.maximum(-z, -SIGMOID_CLAMP), SIGMOID_CLAMP).astype(np.float32)
    e = exp_f32(t)
    return (np.float32(1.0) / (np.float32(1.0) + e)).astype(np.float32)


def router_logits(x: np.ndarray, wr: np.ndarray) -> np.ndarray:
    """x fp32 [T, H] and wr fp32 [E, H] (bf16-exact values) -> logits fp32 [T, E], fixed order."""
    x = np.asarray(x, dtype=np.float32)
    wr = np.asarray(wr, dtype=np.float32)
    t_, h_ = x.shape
    e_ = wr.shape[0]
    assert h_ % ROUTER_CHUNK == 0
    acc = np.zeros((t_, e_), dtype=np.float32)
    for c0 in range(0, h_, ROUTER_CHUNK):
        part = np.zeros((t_, e_), dtype=np.float32)
        for h in range(c0, c0 + ROUTER_CHUNK):
            part = part + x[:, h, None] * wr[None, :, h]    # fp32 product (exact), fp32 add
        acc = acc + part
    return acc


@dataclass
class Routing:
    logits: np.ndarray        # fp32 [T, E]
    score: np.ndarray         # fp32 [T, E]
    key: np.ndarray           # fp32 [T, E]
    topk_idx: np.ndarray      # int32 [T, k]
    topk_w: np.ndarray        # fp32 [T, k]
    counts: np.ndarray        # int32 [E]       live slots per expert
    offsets: np.ndarray       # int32 [E + 1]   exclusive scan of counts
    slot_of_row: np.ndarray   # int32 [S]       plan row -> t * k + j
    row_of_slot: np.ndarray   # int32 [T * k]   t * k + j -> plan row, -1 for dead rows


def topk_select(key: np.ndarray, k: int) -> np.ndarray:
    """Rank experts by (key descending, expert index ascending); keep the first k."""
    t_, e_ = key.shape
    out = np.empty((t_, k), dtype=np.int32)
    eidx = np.arange(e_)
    for t in range(t_):
        order = np.lexsort((eidx, -key[t].astype(np.float64)))
        out[t] = order[:k]
    return out


SURVIVAL_THRESHOLD = 0.2


def dead_from_survival(p_survive, threshold: float = SURVIVAL_THRESHOLD) -> np.ndarray:
    """Dead verification rows (post 2, "Speculative decoding"): a draft row whose estimated chance
    of surviving verification is below the threshold (0.2 there) skips the expert weight reads.
    Compared in fp32, dead = p < threshold: a row exactly at the threshold, and a NaN estimate,
    stay live."""
    p = np.asarray(p_survive, dtype=np.float32)
    return (p < np.float32(threshold)).astype(np.uint8)


def check_anchors(anchor, t_: int) -> np.ndarray | None:
    """anchor[t] = -1 (route row t itself) or the index a of a row routed by itself (anchor[a] = -1).
    TP4 serving profile README ("DeepSeek-V4.1-Flash-4x-DGX-Spark-TP4"), settings table row
    "Verify length": verify rows the confidence head does not expect to survive reuse the anchor
    row's experts inside the router, so they read no extra expert weights."""
    if anchor is None:
        return None
    a = np.asarray(anchor, dtype=np.int64)
    if a.shape != (t_,):
        raise ValueError("anchor must have one entry per row")
    bad = (a < -1) | (a >= t_)
    if np.any(bad):
        raise ValueError("anchor index out of range")
    ref = a[a >= 0]
    if np.any(a[ref] != -1):
        raise ValueError("an anchor row must route itself")
    return a


def route(x: np.ndarray, wr: np.ndarray, bias: np.ndarray, k: int,
          dead: np.ndarray | None = None, anchor: np.ndarray | None = None) -> Routing:
    """Top-k sigmoid gating; rows with anchor[t] = a >= 0 take row a's experts (in a's rank order)
    and weight them with their own scores: w_j = score[t, e_j] / ((score[t, e_0] + ...) + ...)."""
    logits = router_logits(x, wr)
    score = sigmoid_f32(logits)
    key = (score + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float32)
    idx = topk_select(key, k)
    t_, e_ = key.shape
    a = check_anchors(anchor, t_)
    if a is not None:
        for t in range(t_):
            if a[t] >= 0:
                idx[t] = idx[a[t]]
    sel = np.take_along_axis(score, idx, axis=1)               # fp32 [T, k], rank order
    total = np.zeros(t_, dtype=np.float32)
    for j in range(k):
        total = (total + sel[:, j]).astype(np.float32)
    w = (sel / total[:, None]).astype(np.float32)
    return plan(logits, score, key, idx, w, e_, dead)


def plan(logits, score, key, idx, w, e_, dead) -> Routing:
    t_, k = idx.shape
    live = np.ones(t_, dtype=bool) if dead is None else ~np.asarray(dead, dtype=bool)
    counts = np.zeros(e_, dtype=np.int32)
    for t in range(t_):
        if live[t]:
            for j in range(k):
                counts[idx[t, j]] += 1
    offsets = np.zeros(e_ + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    fill = offsets[:-1].copy()
    slot_of_row = np.zeros(int(offsets[-1]), dtype=np.int32)
    row_of_slot = np.full(t_ * k, -1, dtype=np.int32)
    for e in range(e_):                       # expert-major, then token order
        for t in range(t_):
            if not live[t]:
                continue
            hit = np.nonzero(idx[t] == e)[0]
            for j in hit:
                p = fill[e]
                fill[e] += 1
                slot_of_row[p] = t * k + j
                row_of_slot[t * k + j] = p
    return Routing(logits, score, key, idx, w, counts, offsets, slot_of_row, row_of_slot)


# ----------------------------------------------------------------------------------------------
# Activation quantisation and weight quantisation (MX formats)
# ----------------------------------------------------------------------------------------------
def quant_mxfp8(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """x [R, C] (bf16-exact values) -> E4M3 codes u8 [R, C], UE8M0 bytes u8 [R, C/32]."""
    return F.quantize_blocks(np.asarray(x, dtype=np.float64), "e4m3")


def quant_mxfp4(w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """w fp32 [R, C] -> packed E2M1 u8 [R, C/2] (element 2m in the low nibble), UE8M0 [R, C/32]."""
    codes, s = F.quantize_blocks(np.asarray(w, dtype=np.float64), "e2m1")
    return F.pack_e2m1(codes), s


def decode_mxfp4(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    return F.dequant_blocks(F.decode_e2m1(F.unpack_e2m1(packed)), scales)


def decode_mxfp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    return F.dequant_blocks(F.decode_e4m3(codes), scales)


# ----------------------------------------------------------------------------------------------
# Expert GEMMs
# ----------------------------------------------------------------------------------------------
class ExpertWeights:
    """Canonical MXFP4 weights of one projection for all experts, decoded lazily per expert.

    codes u8 [E, R, K/2] (row-major, K contiguous) and scales u8 [E, R, K/32].
    """

    def __init__(self, codes: np.ndarray, scales: np.ndarray, cache: int = 4):
        self.codes, self.scales = codes, scales
        self._cache: dict[int, np.ndarray] = {}
        self._order: list[int] = []
        self._cap = cache

    def __getitem__(self, e: int) -> np.ndarray:
        if e not in self._cache:
            if len(self._order) >= self._cap:
                self._cache.pop(self._order.pop(0))
            self._cache[e] = decode_mxfp4(self.codes[e], self.scales[e])
            self._order.append(e)
        return self._cache[e]


class DenseWeights:
    """One dense MXFP8 projection (the shared expert): codes u8 [R, K] E4M3 and scales u8 [R, K/32],
    presented like a one-expert ExpertWeights (index 0)."""

    def __init__(self, codes: np.ndarray, scales: np.ndarray):
        self.codes = np.asarray(codes)[None]
        self.scales = np.asarray(scales)[None]
        self._dec = None

    def __getitem__(self, e: int) -> np.ndarray:
        if e != 0:
            raise IndexError("a dense projection has one expert")
        if self._dec is None:
            self._dec = decode_mxfp8(self.codes[0], self.scales[0])
        return self._dec


@dataclass
class SharedExpert:
    """TP4 serving profile README, "Rank-0 decode profile" table (shared expert on a side stream) and
    settings row DSV41_SHARED_PAD_K (the shared expert runs on an MXFP8 kernel): one dense SwiGLU
    expert every live row passes through, weight 1, added after the routed slots."""
    w13: DenseWeights          # [2 I_s, H]: rows 0..I_s-1 gate, I_s..2 I_s-1 up
    w2: DenseWeights           # [H, I_s]
    inter: int                 # I_s


@dataclass
class W13Result:
    a: np.ndarray              # float64 [S, I]  pre-requant SwiGLU, plan order
    a32: np.ndarray            # fp32    [S, I]  the values the requant decisions are taken on
    hq: np.ndarray             # u8      [S, I]
    hs: np.ndarray             # u8      [S, I/32]
    flip_ok: np.ndarray        # bool    [S, I]  code may legitimately differ (near a boundary)


def silu_mul(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g)) * u


def requant_flip_eligible(a: np.ndarray, rel_tol: float) -> np.ndarray:
    """Elements whose E4M3 code could change if a moved by up to the stated tolerance.

    tol = rel_tol * max(|a|, rms of a's row). An element is eligible when the interval
    [a - tol, a + tol] straddles a rounding boundary of its own code, or when its block's amax,
    moved by its own tolerance, crosses a scale boundary (then the whole block may rescale).
    """
    a = np.asarray(a, dtype=np.float64)
    rms = np.sqrt(np.mean(a * a, axis=-1, keepdims=True))
    tol = rel_tol * np.maximum(np.abs(a), rms)
    r, c = a.shape
    ab = np.abs(a).reshape(r, c // F.BLOCK, F.BLOCK)
    tb = tol.reshape(r, c // F.BLOCK, F.BLOCK)
    amax = ab.max(-1)
    amax_tol = np.take_along_axis(tb, ab.argmax(-1)[..., None], -1)[..., 0]
    s_lo = F.scale_exponent(np.maximum(amax - amax_tol, 0.0), F.E4M3_MAX)
    s_hi = F.scale_exponent(amax + amax_tol, F.E4M3_MAX)
    block_flip = np.repeat(s_lo != s_hi, F.BLOCK, axis=-1)
    s = np.repeat(F.scale_exponent(amax, F.E4M3_MAX), F.BLOCK, axis=-1)
    lo = F.encode_e4m3((a - tol) * np.ldexp(1.0, -s))
    hi = F.encode_e4m3((a + tol) * np.ldexp(1.0, -s))
    return block_flip | (lo != hi)


def w13_swiglu(xq: np.ndarray, xs: np.ndarray, w13: ExpertWeights, routing: Routing, k: int,
               inter: int, rows: np.ndarray | None = None, rel_tol: float = 1e-5) -> W13Result:
    """SwiGLU of the gate/up projection for plan rows `rows` (default: every live slot)."""
    s_all = int(routing.offsets[-1])
    rows = np.arange(s_all) if rows is None else np.asarray(rows)
    a = np.zeros((len(rows), inter), dtype=np.float64)
    expert_of_row = np.searchsorted(routing.offsets, rows, side="right") - 1
    for n, p in enumerate(rows):
        slot = routing.slot_of_row[p]
        t = slot // k
        e = int(expert_of_row[n])
        xhat = decode_mxfp8(xq[t], xs[t])
        w = w13[e]
        g = w[:inter] @ xhat
        u = w[inter:] @ xhat
        a[n] = silu_mul(g, u)
    a32 = a.astype(np.float32)
    hq, hs = F.quantize_blocks(a32.astype(np.float64), "e4m3")
    return W13Result(a, a32, hq, hs, requant_flip_eligible(a, rel_tol))


def w2_slots(hq: np.ndarray, hs: np.ndarray, w2: ExpertWeights, routing: Routing, k: int,
             rows: np.ndarray | None = None) -> np.ndarray:
    """Per-slot down projection scaled by the routing weight: float64 [len(rows), H]."""
    s_all = int(routing.offsets[-1])
    rows = np.arange(s_all) if rows is None else np.asarray(rows)
    expert_of_row = np.searchsorted(routing.offsets, rows, side="right") - 1
    h_ = w2.codes.shape[1]
    y = np.zeros((len(rows), h_), dtype=np.float64)
    for n, p in enumerate(rows):
        slot = routing.slot_of_row[p]
        t, j = divmod(int(slot), k)
        e = int(expert_of_row[n])
        hhat = decode_mxfp8(hq[n], hs[n])
        y[n] = np.float64(routing.topk_w[t, j]) * (w2[e] @ hhat)
    return y


def combine_exact(y_by_slot: dict[int, np.ndarray], t_: int, k: int, h_: int, tokens,
                  y_shared: dict[int, np.ndarray] | None = None) -> np.ndarray:
    """((y_0 + y_1) + ...) in float64 for the given tokens, before the output rounding; absent
    slots (dead) give 0. A shared-expert row, when given, is added after the routed slots."""
    out = np.zeros((len(tokens), h_), dtype=np.float64)
    for n, t in enumerate(tokens):
        acc = np.zeros(h_, dtype=np.float64)
        live = False
        for j in range(k):
            yj = y_by_slot.get(t * k + j)
            if yj is not None:
                acc = acc + yj
                live = True
        if live and y_shared is not None and int(t) in y_shared:
            acc = acc + y_shared[int(t)]
        out[n] = acc if live else 0.0
    return out


def combine(y_by_slot: dict[int, np.ndarray], t_: int, k: int, h_: int, tokens) -> np.ndarray:
    """out[t] = bf16(((y_0 + y_1) + ...) ) for the given tokens; absent slots (dead) give +0."""
    return F.round_to_bf16(combine_exact(y_by_slot, t_, k, h_, tokens)) + 0.0   # + 0.0: -0.0 -> +0.0


def shared_expert(xq: np.ndarray, xs: np.ndarray, shared: SharedExpert, tokens) -> tuple[W13Result, np.ndarray]:
    """The shared expert for `tokens`: the same SwiGLU, requantisation and down projection as a
    routed expert (one expert, every token, weight 1). Returns the W13 result (rows in `tokens`
    order) and y float64 [len(tokens), H]."""
    tokens = np.asarray(tokens, dtype=np.int64)
    t_ = len(tokens)
    ident = Routing(None, None, None, np.zeros((t_, 1), np.int32), np.ones((t_, 1), np.float32),
                    np.array([t_], np.int32), np.array([0, t_], np.int32), np.arange(t_, dtype=np.int32),
                    np.arange(t_, dtype=np.int32))
    r13 = w13_swiglu(xq[tokens], xs[tokens], shared.w13, ident, 1, shared.inter)
    y = w2_slots(r13.hq, r13.hs, shared.w2, ident, 1)
    return r13, y


@dataclass
class ForwardResult:
    routing: Routing
    xq: np.ndarray
    xs: np.ndarray
    w13: W13Result
    out: np.ndarray            # float64 values of the bf16 output [len(tokens), H]
    tokens: np.ndarray
    out_exact: np.ndarray      # the same sums before the bf16 rounding


def forward(x, wr, bias, k, w13: ExpertWeights, w2: ExpertWeights, inter: int,
            dead=None, tokens=None, anchor=None, shared: SharedExpert | None = None) -> ForwardResult:
    """The whole layer. With `tokens`, only those output rows (and their slots) are computed;
    routing and quantisation of every row are still computed (they are cheap and row-local)."""
    x = np.asarray(x, dtype=np.float32)
    t_, h_ = x.shape
    routing = route(x, wr, bias, k, dead, anchor)
    xq, xs = quant_mxfp8(x)
    tokens = np.arange(t_) if tokens is None else np.asarray(tokens)
    rows = []
    for t in tokens:
        for j in range(k):
            p = routing.row_of_slot[t * k + j]
            if p >= 0:
                rows.append(p)
    rows = np.array(sorted(rows), dtype=np.int64)
    r13 = w13_swiglu(xq, xs, w13, routing, k, inter, rows)
    y = w2_slots(r13.hq, r13.hs, w2, routing, k, rows)
    y_by_slot = {int(routing.slot_of_row[p]): y[n] for n, p in enumerate(rows)}
    y_sh = None
    if shared is not None:
        live = np.ones(t_, bool) if dead is None else ~np.asarray(dead, bool)
        toks = np.array([t for t in tokens if live[t]], dtype=np.int64)
        if len(toks):
            _, ys = shared_expert(xq, xs, shared, toks)
            y_sh = {int(t): ys[n] for n, t in enumerate(toks)}
    out_exact = combine_exact(y_by_slot, t_, k, h_, tokens, y_sh)
    out = F.round_to_bf16(out_exact) + 0.0
    r13_rows = r13
    r13_rows.rows = rows
    return ForwardResult(routing, xq, xs, r13_rows, out, tokens, out_exact)

"""Plain CPU oracle for the NVFP4 block-scaled MoE expert path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` use it.  It shares no code,
tables or constants with the CUDA library under
``nvfp4_block_scaled_quant_gb300/csrc``.

Everything here is written to be checked by eye against the definitions:

* quantisation steps run in IEEE fp32 (numpy float32, one rounding per
  operation, no fused multiply-add);
* dequantised operands and every contraction are fp64;
* the routing permutation is the plain counting definition.

Sources (the three commit-log pages of the "nvfp4-megamoe-kernel" project):

* page 2 (commit efe63ca, single_shot_inference.py), the weight_scale_2 fix:
  a weight decodes as lut[w] * weight_scale * weight_scale_2;
* page 1 (commit 1121cd7, single_shot_inference.py), the scale-semantics
  passage: the GEMM is y = (x * scale_a * gsa) @ (w * scale_b * gsb); the
  global scalars of both sides fold into one multiplier;
* page 3 (commit 4c6464e, vllm), the activation global-scale passage: gs =
  amax / (6 * 448) is the dequantisation multiplier, not its inverse;
* page 3, the grouped-GEMM launch contract: int32 expert offsets, padded and
  swizzled A-side scales;
* page 3, the MoE shape rules: the MoE output width is the hidden size.

Readings taken where the pages are silent (each is also listed in the design
notes): E2M1 and E4M3 conversions round to nearest, ties to even, saturating
at the largest finite value; the block scale is fl32(amax_b / fl32(6 * gs));
element codes come from fl32(x * fl32(1 / d)) with d = fl32(dec(sf) * gs);
a block whose d is zero or has no finite fp32 reciprocal encodes as all-zero
codes; the sign of a quotient that rounds to zero is kept (code 0x8); two
codes per byte, element 2j in the low nibble; w13 rows [0, I) are the gate
projection and rows [I, 2I) the up projection; h is re-quantised from fp32
without a bf16 rounding; the shared expert has weight 1; routing ties keep
the flat order f = t * topk + j.

Pins: see tests/test_oracle_pins.py.  The scale-factor swizzle
(``sf_swizzle_offsets``) has only invariant pins on the CPU; the hardware's
own reading of it is what the GPU GEMM parity tests check.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Dict, Optional, Sequence

import numpy as np

# E2M1 magnitudes for codes 0..7 (sign in bit 3): OCP Microscaling Formats
# spec v1.0, FP4 E2M1 element encoding.
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E2M1_MAX = 6.0
E4M3_MAX = 448.0
GS_DIVISOR = np.float32(6.0 * 448.0)  # 2688, exact in fp32
BLOCK = 16  # elements sharing one E4M3 scale

F32 = np.float32


# ---------------------------------------------------------------------------
# Element formats
# ---------------------------------------------------------------------------

def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """Value of 4-bit E2M1 codes (bit 3 = sign, bits 2..0 index the magnitude)."""
    c = np.asarray(codes).astype(np.int64)
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where((c & 8) != 0, -mag, mag)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """Round fp32 values to E2M1 codes: nearest, ties to the even code, saturate at 6.

    The magnitude thresholds are the midpoints between neighbouring grid values
    {0, .5, 1, 1.5, 2, 3, 4, 6}; at a midpoint the even code (mantissa bit 0)
    wins, which gives ``>`` at 0.25, 1.25, 2.5, 5 and ``>=`` at 0.75, 1.75, 3.5.
    The sign bit follows the sign of the input, including for values that
    round to zero (-0.1 -> 0x8).
    """
    v = np.asarray(v, dtype=np.float32)
    m = np.abs(v).astype(np.float64)
    code = ((m > 0.25).astype(np.uint8) + (m >= 0.75) + (m > 1.25) + (m >= 1.75)
            + (m > 2.5) + (m >= 3.5) + (m > 5.0)).astype(np.uint8)
    return code | (np.signbit(v).astype(np.uint8) << 3)


def ue4m3_decode(b: np.ndarray) -> np.ndarray:
    """Value of unsigned E4M3 scale bytes (bias 7, subnormals when exponent is 0)."""
    b = np.asarray(b).astype(np.int64)
    e = (b >> 3) & 15
    m = b & 7
    sub = m.astype(np.float64) * 2.0 ** -9
    norm = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    return np.where(e == 0, sub, norm)


def ue4m3_encode(s: np.ndarray) -> np.ndarray:
    """Round non-negative fp32 values to E4M3 bytes: nearest-even, saturate at 448 (0x7E)."""
    s = np.asarray(s, dtype=np.float32).astype(np.float64)
    out = np.zeros(s.shape, dtype=np.int64)
    sat = s >= E4M3_MAX
    small = s < 2.0 ** -6
    # subnormal range: the value is m * 2^-9 with m in 0..7 (m == 8 is 2^-6, code 0x08)
    out = np.where(small, np.rint(np.where(small, s, 0.0) * 2.0 ** 9).astype(np.int64), out)
    # normal range 2^-6 <= s < 448: s = f * 2^e with 1 <= f < 2
    with np.errstate(divide="ignore", invalid="ignore"):
        mant, ex = np.frexp(np.where(small | sat, 1.0, s))
    e = ex - 1
    f = mant * 2.0
    m = np.rint((f - 1.0) * 8.0).astype(np.int64)
    carry = m == 8
    e = np.where(carry, e + 1, e)
    m = np.where(carry, 0, m)
    normal = ((e + 7) << 3) | m
    out = np.where(~small & ~sat, normal, out)
    out = np.where(sat, 0x7E, out)
    return np.minimum(out, 0x7E).astype(np.uint8)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 (exact)."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 bit patterns, nearest-even (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


# ---------------------------------------------------------------------------
# NVFP4 block quantisation (activations and weights alike)
# ---------------------------------------------------------------------------

def global_scale(x: np.ndarray) -> np.float32:
    """gs = fl32(amax / (6 * 448)) over the whole tensor (page 3, activation global scale)."""
    amax = F32(np.max(np.abs(np.asarray(x, dtype=np.float32)))) if np.size(x) else F32(0.0)
    return F32(amax / GS_DIVISOR)


@dataclass
class Quantized:
    codes: np.ndarray  # (M, K) uint8, one 4-bit code per element
    sf: np.ndarray     # (M, K/16) uint8 E4M3 block scales, row-major
    gs: np.float32     # global dequantisation multiplier


def quantize(x: np.ndarray, gs: Optional[float] = None) -> Quantized:
    """Quantise a (M, K) fp32 tensor to NVFP4 with global scale gs.

    Per block b of 16 consecutive elements along K:
      s   = fl32(amax_b / fl32(6 * gs))         (0 when 6 * gs is 0)
      sf  = E4M3(s)
      d   = fl32(dec(sf) * gs)
      r   = fl32(1 / d)
      q_i = E2M1(fl32(x_i * r))                 (all codes 0 when d == 0 or r is inf)
    With ``gs=None`` the dynamic global scale of the tensor is used.
    """
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 16")
    g = global_scale(x) if gs is None else F32(gs)
    xb = x.reshape(M, K // BLOCK, BLOCK)
    amax_b = np.max(np.abs(xb), axis=2)
    six_gs = F32(F32(6.0) * g)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        s = (amax_b / six_gs).astype(np.float32) if six_gs != 0 else np.zeros_like(amax_b)
        sf = ue4m3_encode(s)
        d = (ue4m3_decode(sf).astype(np.float32) * g).astype(np.float32)
        r = (F32(1.0) / d).astype(np.float32)
        zero_block = (d == 0) | np.isinf(r)
        q = (xb * r[:, :, None]).astype(np.float32)
    codes = e2m1_encode(q)
    codes = np.where(zero_block[:, :, None], np.uint8(0), codes).astype(np.uint8)
    return Quantized(codes.reshape(M, K), sf, g)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """Two codes per byte, element 2j in the low nibble: (M, K) -> (M, K/2)."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 15) | ((c[..., 1::2] & 15) << 4)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 15
    out[..., 1::2] = p >> 4
    return out


def dequantize(codes: np.ndarray, sf: np.ndarray, g: float) -> np.ndarray:
    """value = e2m1(code) * dec(sf) * g in fp64 (page 2: lut[w] * weight_scale * weight_scale_2)."""
    codes = np.asarray(codes)
    M, K = codes.shape
    scale = np.repeat(ue4m3_decode(sf), BLOCK, axis=1)[:, :K]
    return e2m1_decode(codes) * scale * float(g)


# ---------------------------------------------------------------------------
# Tensor-core scale-factor layout (padded 128-row x 4-column blocks)
# ---------------------------------------------------------------------------

def sf_padded_shape(rows: int, K: int):
    kb = K // BLOCK
    return ((rows + 127) // 128) * 128, ((kb + 3) // 4) * 4


def sf_bytes(rows: int, K: int) -> int:
    r, c = sf_padded_shape(rows, K)
    return r * c


def sf_swizzle_offsets(rows: int, K: int) -> np.ndarray:
    """Byte offset of scale (r, c) in the swizzled buffer, for every padded (r, c).

    Rows are grouped by 128 and scale columns by 4; each such 128 x 4 group is a
    contiguous 512-byte block, blocks ordered row-group-major.  Inside a block,
    row r's four scales sit together at byte (r % 32) * 16 + ((r % 128) // 32) * 4.
    """
    R, C = sf_padded_shape(rows, K)
    r = np.arange(R)[:, None]
    c = np.arange(C)[None, :]
    return ((r // 128) * (C // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)


def swizzle_sf(sf: np.ndarray, K: int) -> np.ndarray:
    rows = sf.shape[0]
    R, C = sf_padded_shape(rows, K)
    padded = np.zeros((R, C), dtype=np.uint8)
    padded[:rows, : sf.shape[1]] = sf
    out = np.zeros(R * C, dtype=np.uint8)
    out[sf_swizzle_offsets(rows, K)] = padded
    return out


def unswizzle_sf(buf: np.ndarray, rows: int, K: int) -> np.ndarray:
    off = sf_swizzle_offsets(rows, K)
    full = np.asarray(buf, dtype=np.uint8)[off]
    return full[:rows, : K // BLOCK]


# ---------------------------------------------------------------------------
# RMSNorm feeding the activation quantiser
# ---------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float):
    """RMSNorm of each row: y = x / sqrt(mean(x^2) + eps) * gamma, in fp64.

    Returns (y rounded to bf16 through fp32, as fp32 values; y in fp64; inv_rms fp64).  The
    normalised activations that feed the NVFP4 quantiser are bf16, as the unfused path of page 1
    (the fused-RMSNorm A/B passage) hands x_normed to the quantiser.
    """
    x64 = np.asarray(x, dtype=np.float64)
    inv = 1.0 / np.sqrt(np.mean(x64 * x64, axis=1) + eps)
    y = x64 * inv[:, None] * np.asarray(gamma, dtype=np.float64)[None, :]
    yb = bf16_bits_to_f32(f32_to_bf16_bits(y.astype(np.float32)))
    return yb, y, inv


# ---------------------------------------------------------------------------
# Dense NVFP4 linear
# ---------------------------------------------------------------------------

def linear(xq: Quantized, w_codes: np.ndarray, w_sf: np.ndarray, ws2: float) -> np.ndarray:
    """y[m, n] = sum_k deq(xq)[m, k] * deq(W)[n, k] in fp64.

    The activation side carries gs, the weight side ws2 only (page 2, the input_scale
    passage: the checkpoint input_scale stays off the weight side).
    """
    a = dequantize(xq.codes, xq.sf, xq.gs)
    b = dequantize(w_codes, w_sf, ws2)
    return a @ b.T


def grouped_linear(xq: Quantized, w_codes: Sequence[np.ndarray], w_sf: Sequence[np.ndarray],
                   ws2: Sequence[float]) -> np.ndarray:
    """Fixed-group linear: the input features split into G equal groups, group g of x times W_g.

    y[:, g*N:(g+1)*N] = deq(xq[:, g*K:(g+1)*K]) @ deq(W_g)^T with W_g's own ws2 and the
    activation's single gs (page 3, the wo_a o-projection passage: wo_a is
    a per-group BMM with in_features 4096 per group; the ScaledGroupedGemm passage:
    an NVFP4 grouped linear with n_local_groups = 8).
    """
    G = len(w_codes)
    K = xq.codes.shape[1] // G
    outs = []
    for g in range(G):
        xg = Quantized(xq.codes[:, g * K:(g + 1) * K], xq.sf[:, g * (K // BLOCK):(g + 1) * (K // BLOCK)], xq.gs)
        outs.append(linear(xg, w_codes[g], w_sf[g], ws2[g]))
    return np.concatenate(outs, axis=1)


# ---------------------------------------------------------------------------
# Router gate (FP8-E4M3 round trip of the gate weight, linear, softmax, top-k)
# ---------------------------------------------------------------------------

def e4m3_encode_signed(v: np.ndarray) -> np.ndarray:
    """Signed E4M3 (FN) byte: sign bit 7 plus the unsigned nearest-even, saturating encoding of |v|."""
    v = np.asarray(v, dtype=np.float32)
    return ue4m3_encode(np.abs(v)) | (np.signbit(v).astype(np.uint8) << 7)


def e4m3_decode_signed(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b).astype(np.int64)
    mag = ue4m3_decode(b & 0x7F)
    return np.where((b & 0x80) != 0, -mag, mag)


def router_weight(w_codes: np.ndarray, w_sf: np.ndarray, ws2: float) -> np.ndarray:
    """Gate weight as the router uses it (page 1, the router-gate FP8 round-trip passage):
    dequantise the NVFP4 checkpoint to bf16, quantise to FP8-E4M3 with one per-tensor scale
    s = amax / 448, dequantise back to bf16.  Steps in fp32:
      w  = bf16(fl32(fl32(e2m1 * e4m3) * ws2))
      s  = fl32(amax(|w|) / 448),  q = E4M3(fl32(w * fl32(1 / s)))   (all zero when s == 0)
      wg = bf16(fl32(e4m3(q) * s))
    Returns wg as fp32 values (exactly bf16-representable).
    """
    scale = np.repeat(ue4m3_decode(w_sf), BLOCK, axis=1)[:, : w_codes.shape[1]].astype(np.float32)
    prod = (e2m1_decode(w_codes).astype(np.float32) * scale).astype(np.float32)
    w = bf16_bits_to_f32(f32_to_bf16_bits((prod * F32(ws2)).astype(np.float32)))
    amax = F32(np.max(np.abs(w))) if w.size else F32(0)
    s = F32(amax / F32(448.0))
    if s == 0:
        return np.zeros_like(w)
    r = F32(F32(1.0) / s)
    q = e4m3_encode_signed((w * r).astype(np.float32))
    deq = (e4m3_decode_signed(q).astype(np.float32) * s).astype(np.float32)
    return bf16_bits_to_f32(f32_to_bf16_bits(deq))


def router(x: np.ndarray, wg: np.ndarray, topk: int):
    """Dense router: logits = x @ wg^T (fp64), softmax over the experts, top-k (ties to the
    lower expert id), weights renormalised over the k chosen.  Returns (ids, weights, probs)."""
    logits = np.asarray(x, dtype=np.float64) @ np.asarray(wg, dtype=np.float64).T
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :topk]
    w = np.take_along_axis(p, order, axis=1)
    return order.astype(np.int32), w / w.sum(axis=1, keepdims=True), p


# ---------------------------------------------------------------------------
# Routing
# ---------------------------------------------------------------------------

@dataclass
class Routing:
    counts: np.ndarray      # (E,) int32
    offsets: np.ndarray     # (E+1,) int32, exclusive prefix sum of counts
    sorted_idx: np.ndarray  # (T*k,) int32, flat indices grouped by expert
    inv_idx: np.ndarray     # (T*k,) int32, position of each flat index in sorted_idx


def route(ids: np.ndarray, E: int) -> Routing:
    """Group the flat (token, slot) indices f = t*k + j by expert id.

    counts[e] is the number of f with ids[f] == e; offsets is their exclusive
    prefix sum; within an expert the flat indices keep increasing order, and
    experts appear in increasing id.  Written as the counting definition.
    """
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    counts = [0] * E
    for e in flat:
        if not 0 <= e < E:
            raise ValueError(f"expert id {e} outside [0, {E})")
        counts[e] += 1
    offsets = [0] * (E + 1)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    cursor = list(offsets[:E])
    sorted_idx = [0] * len(flat)
    inv_idx = [0] * len(flat)
    for f, e in enumerate(flat):
        sorted_idx[cursor[e]] = f
        inv_idx[f] = cursor[e]
        cursor[e] += 1
    i32 = np.int32
    return Routing(np.array(counts, i32), np.array(offsets, i32),
                   np.array(sorted_idx, i32), np.array(inv_idx, i32))


# ---------------------------------------------------------------------------
# MoE expert computation
# ---------------------------------------------------------------------------

def silu(g: np.ndarray) -> np.ndarray:
    """SiLU(g) = g / (1 + exp(-g)), fp64."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


@dataclass
class Expert:
    """One expert in checkpoint layout: codes (N, K) unpacked, sf (N, K/16), ws2."""
    w13_codes: np.ndarray  # (2I, H): rows [0, I) gate, [I, 2I) up
    w13_sf: np.ndarray
    w13_ws2: float
    w2_codes: np.ndarray   # (H, I)
    w2_sf: np.ndarray
    w2_ws2: float


@dataclass
class ExpertResult:
    h: np.ndarray       # (rows, I) fp64 SiLU(gate) * up
    hq: Quantized       # h re-quantised with the static a2 global scale
    o: np.ndarray       # (rows, H) fp64 down-projection output


def expert_forward(xq_rows: Quantized, ex: Expert, a2_gs: float) -> ExpertResult:
    """One expert on a set of quantised token rows: w13 -> SiLU(gate)*up -> re-quant -> w2."""
    gu = linear(xq_rows, ex.w13_codes, ex.w13_sf, ex.w13_ws2)
    I = gu.shape[1] // 2
    h = silu(gu[:, :I]) * gu[:, I:]
    hq = quantize(h.astype(np.float32), gs=a2_gs)
    o = expert_w2(hq, ex)
    return ExpertResult(h, hq, o)


def expert_w2(hq: Quantized, ex: Expert) -> np.ndarray:
    return linear(hq, ex.w2_codes, ex.w2_sf, ex.w2_ws2)


@dataclass
class MoEResult:
    y: np.ndarray                 # (len(tokens), H) fp64
    xq: Quantized                 # quantised activations of all T tokens
    routing: Routing
    rows: Dict[tuple, ExpertResult]  # (token, slot) -> per-row result; slot -1 = shared


def _expert_job(job) -> ExpertResult:
    """One expert's share of the MoE: ``job`` = (expert or expert source, expert id, the
    quantised rows routed to it, its static a2 scale).  Module level so a process pool can run it."""
    src, e, xq_rows, a2 = job
    ex = src if isinstance(src, Expert) else src(e)
    return expert_forward(xq_rows, ex, a2)


def moe_forward(x: np.ndarray, ids: np.ndarray, topk_w: np.ndarray,
                experts: Callable[[int], Expert], E: int, a2_gs: Sequence[float],
                shared: Optional[Expert] = None, a1_gs: Optional[float] = None,
                tokens: Optional[Sequence[int]] = None, mapper=map) -> MoEResult:
    """Routed MoE with an optional always-active shared expert.

    For each token t and slot j with e = ids[t, j]:
        y[t] += topk_w[t, j] * W2_e( requant( SiLU(gate_e(xq[t])) * up_e(xq[t]) ) )
    plus the shared expert with weight 1.  xq uses one global scale over all T
    tokens (dynamic amax/2688 unless ``a1_gs`` is given); the re-quantisation
    of h uses the static per-expert scale a2_gs[e] (a2_gs[E] for the shared
    expert).  ``tokens`` restricts the output rows computed (all by default);
    the global scale and routing always cover all T tokens.

    The rows routed to one expert go through that expert together (its weights
    are dequantised once); every row's result is the same per-row definition.
    ``mapper`` (the builtin ``map`` by default, or a process pool's ``imap``)
    runs the per-expert jobs; ``experts`` must then be picklable.  Each token's
    sum is taken in slot order, then the shared expert.
    """
    x = np.asarray(x, dtype=np.float32)
    T, H = x.shape
    k = ids.shape[1]
    xq = quantize(x, gs=a1_gs)
    routing = route(ids, E)
    toks = list(range(T)) if tokens is None else [int(t) for t in tokens]
    slots_of: Dict[int, list] = {}
    for t in toks:
        for j in range(k):
            slots_of.setdefault(int(ids[t, j]), []).append((t, j))
    jobs = [(experts, e, slots_of[e]) for e in sorted(slots_of)]
    if shared is not None:
        jobs.append((shared, E, [(t, -1) for t in toks]))

    def payload(job):
        src, e, slots = job
        ts = [t for t, _ in slots]
        return src, e, Quantized(xq.codes[ts], xq.sf[ts], xq.gs), a2_gs[e]

    rows: Dict[tuple, ExpertResult] = {}
    for (_, _, slots), res in zip(jobs, mapper(_expert_job, [payload(jb) for jb in jobs])):
        for r, s in enumerate(slots):
            rows[s] = ExpertResult(res.h[r:r + 1], Quantized(res.hq.codes[r:r + 1], res.hq.sf[r:r + 1], res.hq.gs),
                                   res.o[r:r + 1])
    y = np.zeros((len(toks), H), dtype=np.float64)
    for i, t in enumerate(toks):
        for j in range(k):
            y[i] += float(topk_w[t, j]) * rows[(t, j)].o[0]
        if shared is not None:
            y[i] += rows[(t, -1)].o[0]
    return MoEResult(y, xq, routing, rows)


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))

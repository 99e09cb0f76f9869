"""Plain CPU oracle for the AWQ W4A16 group-quantized linear layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this module.  The
product library never calls it, and this module imports nothing from the
product package: the two sides share only the seeded input generator in
``awq_inputs``.

Sources (web pages describing Activation-aware Weight Quantization):

* [P1] "awq-quantization（AWQ量化技术）Skill 是什么？如何下载安装使用？"
  (skillsbot.cn), sections "该技能的主要功能和特点" and "步骤 2/3".
* [P2] "AWQ量化实战：无需重训，把大模型压进4bit显存" (xdnf.cn), §1.1, §2.1-§2.3,
  §3.3, §3.4, §5.1.
* [P4] "大模型量化部署实战：GPTQ与AWQ算法" (yunthe.com), section
  "大模型量化的核心原理与位宽选择".
* [P5] "什么是激活感知权重量化（AWQ）？" (aiboss88.com), section "工作机制".

Everything is written for clarity, not speed: fp32 where the method's
integer decisions are taken (so that a code is decided exactly as the
definition says), fp64 for every sum.  Readings taken where the pages are
silent are marked READING.

Parity status: every function here is pinned by a ``-m "not gpu"`` test
against closed forms, invariants, brute force on tiny inputs or hand-derived
golden values (tests/test_oracle_pins.py).  No function is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

GROUP = 128          # [P1] 步骤 2 quant_config q_group_size; [P2] §2.3
W_BIT = 4            # [P1] 步骤 2 w_bit
QMAX = (1 << W_BIT) - 1
N_GRID = 20          # number of alpha candidates, all in [0, 1)
A_FLOOR = np.float32(1e-8)          # READING: floor on mean|x| before the power
S_MIN = np.float32(2.0 ** -14)      # READING: smallest normal fp16 step
S_MAX = np.float32(65504.0)         # READING: largest finite fp16 step
TOL_REL = 4e-3       # per-element matmul tolerance (relative to sum |x~ w^|)
MSE_REL = 1e-4       # search tolerance on the MSE of the chosen alpha


# ---------------------------------------------------------------- a1: stats
def absmean(X16: np.ndarray) -> np.ndarray:
    """Per-input-channel activation strength ``a_c = mean_t |x_tc|``.

    [P2] §2.1: collect the calibration activations of every input channel,
    take absolute values and average over many tokens (a running mean or a
    plain sum-then-divide are both acceptable).  READING: plain mean, summed
    in fp64, stored as fp32.
    """
    X = np.asarray(X16)
    T = X.shape[0]
    acc = np.zeros(X.shape[1], dtype=np.float64)
    for t0 in range(0, T, 4096):                # bounded memory only
        acc += np.abs(X[t0:t0 + 4096].astype(np.float64)).sum(axis=0)
    return (acc / T).astype(np.float32)


# ------------------------------------------------------- a2: scale candidates
def alpha_grid(n_grid: int = N_GRID) -> np.ndarray:
    """The alpha candidates ``{0, 1/n, ..., (n-1)/n}`` (fp64).

    [P2] §2.2: the scale is found by a grid search over a candidate interval.
    READING: 20 evenly spaced points in [0, 1), starting at 0.
    """
    return np.arange(n_grid, dtype=np.float64) / n_grid


def channel_scales(a: np.ndarray, alpha: float):
    """Activation-aware per-channel scales ``s_c = a_c ** alpha`` and ``1/s_c``.

    [P2] §2.2 and [P5] 工作机制: salient channels (large mean|x|) are scaled
    up by a factor derived from the offline activation statistics.
    READING: ``a`` is floored at 1e-8 (fp32) so that 1/s_c stays finite; the
    power is taken in fp64 and rounded to fp32; no normalisation of s_c.
    ``inv_s`` is the IEEE fp32 quotient ``1 / s_c``.
    """
    a32 = np.maximum(np.asarray(a, dtype=np.float32), A_FLOOR)
    s_c = np.power(a32.astype(np.float64), float(alpha)).astype(np.float32)
    inv_s = (np.float32(1.0) / s_c).astype(np.float32)
    return s_c, inv_s


# --------------------------------------------------- a3: scaled group RTN
def quantize(W16: np.ndarray, s_c: np.ndarray | None = None, group: int = GROUP,
             w_bit: int = W_BIT, zero_point: bool = True):
    """Group round-to-nearest of ``W' = W diag(s_c)``.

    [P2] §1.1 (round to nearest), §2.1 (the channel is the input dimension;
    the weight is out x in and is grouped along the input dimension), §2.3
    (``group`` consecutive input channels share one step: 128, also 64 or
    32), [P4] (a scale plus a zero point per group), [P1] 步骤 2 (zero_point
    on, 4 bits, group 128), [P2] §3.3 (zero_point off is the symmetric form;
    8 bits is the conservative width).

    For each row n and group g (fp32 arithmetic), with qmax = 2^w_bit - 1:

    asymmetric (zero_point on):
      mn, mx = min, max of the group of w'                 (READING: plain)
      s32    = (mx - mn) / qmax, clamped to [2^-14, 65504] (READING)
      s      = fp16_rne(s32)            (the stored scale; codes use it)
      z      = clamp(rint(-mn / s), 0, qmax)
      q      = clamp(rint(w' / s) + z, 0, qmax)
    symmetric (zero_point off), h = 2^(w_bit - 1):
      s32    = max |w'| / (h - 1), clamped to [2^-14, 65504]
      q      = clamp(rint(w' / s), -h, h - 1) + h,   z = h
      READING: [P4] gives the signed range -8..7 for int4; the codes are
      stored offset by h (unsigned), so the stored zero point is the
      constant h and dequantization is the same (q - z) * s.
    with ``rint`` = round half to even and IEEE fp32 division.

    Returns ``q`` uint8 [N, K], ``z`` uint8 [N, G], ``s16`` float16 [N, G].
    """
    assert w_bit in (4, 8) and group in (32, 64, 128)
    qmax = (1 << w_bit) - 1
    W = np.asarray(W16, dtype=np.float16).astype(np.float32)
    N, K = W.shape
    assert K % group == 0, "K must be a multiple of the group size"
    if s_c is not None:
        W = (W * np.asarray(s_c, dtype=np.float32)[None, :]).astype(np.float32)
    G = K // group
    Wg = W.reshape(N, G, group)
    if zero_point:
        mn = Wg.min(axis=2)
        mx = Wg.max(axis=2)
        s32 = ((mx - mn) / np.float32(qmax)).astype(np.float32)
    else:
        h = 1 << (w_bit - 1)
        s32 = (np.abs(Wg).max(axis=2) / np.float32(h - 1)).astype(np.float32)
    s32 = np.minimum(np.maximum(s32, S_MIN), S_MAX)
    s16 = s32.astype(np.float16)
    s = s16.astype(np.float32)
    if zero_point:
        z = np.clip(np.rint((-mn) / s), 0, qmax).astype(np.float32)
        q = np.clip(np.rint(Wg / s[:, :, None]) + z[:, :, None], 0, qmax)
    else:
        z = np.full((N, G), float(h), dtype=np.float32)
        q = np.clip(np.rint(Wg / s[:, :, None]), -h, h - 1) + h
    return (q.reshape(N, K).astype(np.uint8), z.astype(np.uint8), s16)


# ------------------------------------------------------------ packing layout
def pack_codes(q: np.ndarray, w_bit: int = W_BIT) -> np.ndarray:
    """``32 / w_bit`` codes per uint32: ``qweight[n, j]`` holds k = c j + i in
    bits [w_bit i, w_bit (i + 1)) with c = 32 / w_bit (8 nibbles or 4 bytes).

    [P5] 典型例子 names platform-aware weight packing without fixing a
    layout; this layout is the library's documented canonical one.
    """
    c = 32 // w_bit
    q = np.asarray(q, dtype=np.uint32)
    N, K = q.shape
    q = q.reshape(N, K // c, c)
    out = np.zeros((N, K // c), dtype=np.uint32)
    for i in range(c):
        out |= q[:, :, i] << np.uint32(w_bit * i)
    return out


def unpack_codes(qweight: np.ndarray, w_bit: int = W_BIT) -> np.ndarray:
    c = 32 // w_bit
    qw = np.asarray(qweight, dtype=np.uint32)
    N, J = qw.shape
    out = np.empty((N, J, c), dtype=np.uint8)
    for i in range(c):
        out[:, :, i] = (qw >> np.uint32(w_bit * i)) & np.uint32((1 << w_bit) - 1)
    return out.reshape(N, J * c)


def pack_zeros(z: np.ndarray, w_bit: int = W_BIT) -> np.ndarray:
    """Zero points packed like the codes: group g = c j + i in field i;
    pad fields = 0."""
    c = 32 // w_bit
    z = np.asarray(z, dtype=np.uint32)
    N, G = z.shape
    J = (G + c - 1) // c
    zp = np.zeros((N, J * c), dtype=np.uint32)
    zp[:, :G] = z
    return pack_codes(zp, w_bit)


def unpack_zeros(zeros: np.ndarray, G: int, w_bit: int = W_BIT) -> np.ndarray:
    return unpack_codes(zeros, w_bit)[:, :G]


def awq_pack(W16: np.ndarray, s_c: np.ndarray | None = None, group: int = GROUP,
             w_bit: int = W_BIT, zero_point: bool = True):
    """Quantize and pack: returns ``qweight`` uint32 [N, K w_bit / 32],
    ``scales`` float16 [N, K/group], ``zeros`` uint32 [N, ceil(G w_bit / 32)]."""
    q, z, s16 = quantize(W16, s_c, group, w_bit, zero_point)
    return pack_codes(q, w_bit), s16, pack_zeros(z, w_bit)


# ------------------------------------------------------------ a4: dequant
def dequant(qweight: np.ndarray, scales: np.ndarray, zeros: np.ndarray,
            group: int = GROUP, w_bit: int = W_BIT) -> np.ndarray:
    """``w^' = (q - z) * s`` in fp32 (exact: a (w_bit+1)-bit integer times an
    fp16).

    [P4]: the integer code is mapped back with its group's scale and zero point.
    """
    q = unpack_codes(qweight, w_bit).astype(np.float32)
    N, K = q.shape
    G = K // group
    z = unpack_zeros(zeros, G, w_bit).astype(np.float32)
    s = np.asarray(scales, dtype=np.float16).astype(np.float32)
    qg = q.reshape(N, G, group)
    return ((qg - z[:, :, None]) * s[:, :, None]).reshape(N, K).astype(np.float32)


# ------------------------------------------------------ a7/a8: the linear
def scaled_activations(X16: np.ndarray, inv_s: np.ndarray | None) -> np.ndarray:
    """``x~ = fp32(x) * (1/s_c)`` rounded to fp32: the equivalent transformation
    puts ``diag(1/s_c)`` on the activations ([P2] §2.2, [P5] 工作机制)."""
    X = np.asarray(X16, dtype=np.float16).astype(np.float32)
    if inv_s is None:
        return X
    return (X * np.asarray(inv_s, dtype=np.float32)[None, :]).astype(np.float32)


def linear(X16, qweight, scales, zeros, inv_s=None, group: int = GROUP, w_bit: int = W_BIT):
    """``Y^ = (X diag(1/s_c)) W^'^T`` summed in fp64.

    Returns ``(Y, B)``: ``Y`` fp64 [M, N] and the tolerance base
    ``B[m, n] = sum_k |x~_mk * w^'_nk|`` (fp64).
    """
    xt = scaled_activations(X16, inv_s).astype(np.float64)
    wq = dequant(qweight, scales, zeros, group, w_bit).astype(np.float64)
    return xt @ wq.T, np.abs(xt) @ np.abs(wq).T


def ulp_fp16(y: np.ndarray) -> np.ndarray:
    """Spacing of fp16 numbers at |y| (2^-24 in the subnormal range)."""
    a = np.abs(np.asarray(y, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -24)))
    return np.exp2(np.maximum(e, -14.0) - 10.0)


def tolerance(y_ref: np.ndarray, base: np.ndarray) -> np.ndarray:
    """Per-element bound ``4e-3 * sum_k |x~ w^| + 1 fp16 ulp of y_ref``."""
    return TOL_REL * np.asarray(base, dtype=np.float64) + ulp_fp16(y_ref)


# --------------------------------------------------- a5/a6: alpha search
def _reference_output(X16, W16, rows, t0, t1):
    X = np.asarray(X16[t0:t1], dtype=np.float16).astype(np.float64)
    Wr = np.asarray(W16, dtype=np.float16)[rows].astype(np.float64)
    return X @ Wr.T


def row_errors(X16, W16, s_c, inv_s, rows=None, token_chunk=4096, **cfg):
    """Per-output-row squared error ``e_n = sum_t (Y^_tn - Y_tn)^2`` (fp64)
    for the scaled quantization of ``W`` with the given ``s_c``/``inv_s``.

    ``Y = X W^T`` is the unquantized layer (READING: the fp16 weights, exact
    sum); ``Y^`` is the quantized layer of :func:`linear`.  Only the listed
    ``rows`` are evaluated (quantization is per row, so a row's codes do not
    depend on the other rows).  The token sum is split into chunks only to
    bound memory.
    """
    W16 = np.asarray(W16, dtype=np.float16)
    N = W16.shape[0]
    rows = np.arange(N) if rows is None else np.asarray(rows)
    qw, sc, zs = awq_pack(W16[rows], s_c, **cfg)
    wq = dequant(qw, sc, zs, cfg.get("group", GROUP), cfg.get("w_bit", W_BIT)).astype(np.float64)
    T = X16.shape[0]
    err = np.zeros(len(rows), dtype=np.float64)
    for t0 in range(0, T, token_chunk):
        t1 = min(T, t0 + token_chunk)
        xt = scaled_activations(X16[t0:t1], inv_s).astype(np.float64)
        r = xt @ wq.T - _reference_output(X16, W16, rows, t0, t1)
        err += (r * r).sum(axis=0)
    return err


def search(X16, W16, n_grid: int = N_GRID, rows=None, a=None, **cfg):
    """Activation-aware scale search over ``alpha`` ([P2] §2.2, §3.3 第四步,
    §5.1; [P5] 工作机制: no backpropagation, one coefficient per layer).

    For each alpha_i in :func:`alpha_grid`: s_c = a^alpha_i, quantize
    ``W diag(s_c)``, run the quantized layer on the calibration tokens and
    score ``mse_i = sum (Y^ - Y)^2 / (T * N_rows)``.  alpha* = argmin, ties
    broken by the smallest alpha (first index).

    Returns a dict with ``mse`` [n_grid], ``row_err`` [n_grid, N_rows],
    ``best`` (index), ``alpha``, ``s_c`` and ``inv_s`` of the best candidate.
    """
    X16 = np.asarray(X16, dtype=np.float16)
    if a is None:
        a = absmean(X16)
    T = X16.shape[0]
    W16 = np.asarray(W16, dtype=np.float16)
    rows = np.arange(W16.shape[0]) if rows is None else np.asarray(rows)
    alphas = alpha_grid(n_grid)
    row_err = np.zeros((n_grid, len(rows)), dtype=np.float64)
    for i, al in enumerate(alphas):
        s_c, inv_s = channel_scales(a, al)
        row_err[i] = row_errors(X16, W16, s_c, inv_s, rows, **cfg)
    mse = row_err.sum(axis=1) / (T * len(rows))
    best = int(np.argmin(mse))
    s_c, inv_s = channel_scales(a, alphas[best])
    return {"mse": mse, "row_err": row_err, "best": best,
            "alpha": float(alphas[best]), "s_c": s_c, "inv_s": inv_s, "a": a}


def gram(X16, token_chunk=4096) -> np.ndarray:
    """``H = X^T X`` in fp64 (K x K)."""
    X16 = np.asarray(X16, dtype=np.float16)
    K = X16.shape[1]
    H = np.zeros((K, K), dtype=np.float64)
    for t0 in range(0, X16.shape[0], token_chunk):
        X = X16[t0:t0 + token_chunk].astype(np.float64)
        H += X.T @ X
    return H


def row_errors_gram(H, W16, s_c, inv_s, rows=None, **cfg):
    """Second route to :func:`row_errors` through the identity
    ``sum_t r_tn^2 = d_n^T H d_n`` with ``d_n = inv_s * w^'_n - w_n`` and
    ``H = X^T X``.  Exact in real arithmetic when ``x~ = x * inv_s``; the
    fp32 rounding of ``x~`` in :func:`row_errors` makes the two differ by a
    few 1e-7 relative."""
    W16 = np.asarray(W16, dtype=np.float16)
    rows = np.arange(W16.shape[0]) if rows is None else np.asarray(rows)
    qw, sc, zs = awq_pack(W16[rows], s_c, **cfg)
    wq = dequant(qw, sc, zs, cfg.get("group", GROUP), cfg.get("w_bit", W_BIT)).astype(np.float64)
    d = wq * np.asarray(inv_s, dtype=np.float64)[None, :] - W16[rows].astype(np.float64)
    return np.einsum("nk,kj,nj->n", d, H, d, optimize=True)


# ------------------------------------- fused projections sharing one input
# [P1] 主要功能和特点 (融合模块加速: fused attention / MLP modules) and [P5]
# (TinyChat's kernel fusion): the projections that read the same input are
# one concatenated weight, and the MLP's gate and up projections feed
# SiLU(gate) * up.  READING: the fused gate/up weight stacks the I gate rows
# first and the I up rows after them ([2I, K]), and the product is formed from
# the two projections' exact sums (fp64 here) before the single rounding of
# the output.
SILU_LIP = 1.0999   # max |d silu / dx| = 1.09984 (at x = 2.3994), rounded up


def silu(x):
    """``silu(x) = x / (1 + exp(-x))`` in fp64."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def silu_mul_linear(X16, qweight, scales, zeros, inv_s=None, group: int = GROUP,
                    w_bit: int = W_BIT):
    """``Y = silu(X~ W^'_gate^T) * (X~ W^'_up^T)`` for a fused [2I, K] weight.

    Returns ``(Y, tol)``: ``Y`` fp64 [M, I] and a per-element tolerance that
    carries each projection's bound ``e = 4e-3 * sum |x~ w^|`` through the
    product: ``|d(silu(g) u)| <= L e_g (|u| + e_u) + |silu(g)| e_u`` with
    ``L`` = :data:`SILU_LIP`, plus 1 fp16 ulp of Y and 1e-6 relative for the
    fp32 evaluation of silu.
    """
    Y2, B2 = linear(X16, qweight, scales, zeros, inv_s, group, w_bit)
    two_i = Y2.shape[1]
    assert two_i % 2 == 0, "the fused weight has an even number of rows"
    I = two_i // 2
    g, u = Y2[:, :I], Y2[:, I:]
    eg, eu = TOL_REL * B2[:, :I], TOL_REL * B2[:, I:]
    sg = silu(g)
    Y = sg * u
    tol = SILU_LIP * eg * (np.abs(u) + eu) + np.abs(sg) * eu + ulp_fp16(Y) + 1e-6 * np.abs(Y)
    return Y, tol


# ------------------------------- equivalent transformation into the input op
def fold_inv_scales(W16, inv_s):
    """Fold ``diag(1/s_c)`` into the operator that produces the layer's input.

    [P5] 工作机制 (等价变换: the salient channels are scaled by an equivalent
    transformation whose factors come from offline activation statistics):
    ``(x diag(1/s_c)) (W diag(s_c))^T = x W^T``, so ``1/s_c`` can live in the
    previous operator instead of a runtime multiply.  ``W16`` holds one row per
    input channel of the quantized layer: a norm's weight vector ([K] or
    [K, 1]) or the output rows of the previous linear ([K, C]).  Row k is
    multiplied by ``inv_s[k]`` in fp32 and rounded to fp16 (RNE).
    """
    W = np.asarray(W16, dtype=np.float16)
    shape = W.shape
    W2 = W.reshape(shape[0], -1).astype(np.float32)
    out = (W2 * np.asarray(inv_s, dtype=np.float32)[:, None]).astype(np.float32)
    return out.astype(np.float16).reshape(shape)


# ------------------------------------------------------- weight clipping
# The pages name a clipping parameter (``clip_steps``, suggested 200, in the
# troubleshooting section of "AWQ量化实战..." §5.1) and nothing more.
# READING: after the scale search, each group's range [min, max] of the
# scaled weights may shrink to [r min, r max] with r on a grid
# r_i = 1 - 0.5 i / n (i = 0 .. n-1, n = the number of clip steps); the
# group is quantized from the shrunk range (codes clamp, which clips), and
# the ratio that minimises the group's output error on the calibration
# tokens, e = sum_t (sum_k x~_tk (w^_k - w'_k))^2 = d^T H_g d with
# H_g = X~_g^T X~_g, is kept (ties: the smallest i, the least clipping).
CLIP_MIN = 0.5


def clip_ratios(n_clip: int) -> np.ndarray:
    """``r_i = fp32(1 - 0.5 i / n)``, i = 0..n-1."""
    return (1.0 - CLIP_MIN * np.arange(n_clip, dtype=np.float64) / n_clip).astype(np.float32)


def quantize_clipped(W16, s_c, ratio_idx, n_clip, group=GROUP, w_bit=W_BIT, zero_point=True):
    """:func:`quantize` with each group's range shrunk by ``r[ratio_idx[n, g]]``.

    The shrunk range is ``[fp32(r mn), fp32(r mx)]`` (symmetric: ``r max|w'|``);
    step, zero point and codes follow from it by the same rules (codes clamp,
    which clips the weights outside the range).  ``ratio_idx`` all 0 is
    :func:`quantize` exactly.
    """
    qmax = (1 << w_bit) - 1
    W = np.asarray(W16, dtype=np.float16).astype(np.float32)
    N, K = W.shape
    if s_c is not None:
        W = (W * np.asarray(s_c, dtype=np.float32)[None, :]).astype(np.float32)
    G = K // group
    Wg = W.reshape(N, G, group)
    r = clip_ratios(n_clip)[np.asarray(ratio_idx, dtype=np.int64)]   # fp32 [N, G]
    if zero_point:
        mn = (Wg.min(axis=2) * r).astype(np.float32)
        mx = (Wg.max(axis=2) * r).astype(np.float32)
        s32 = ((mx - mn) / np.float32(qmax)).astype(np.float32)
    else:
        h = 1 << (w_bit - 1)
        s32 = ((np.abs(Wg).max(axis=2) * r).astype(np.float32) / np.float32(h - 1)).astype(np.float32)
    s32 = np.minimum(np.maximum(s32, S_MIN), S_MAX)
    s16 = s32.astype(np.float16)
    s = s16.astype(np.float32)
    if zero_point:
        z = np.clip(np.rint((-mn) / s), 0, qmax).astype(np.float32)
        q = np.clip(np.rint(Wg / s[:, :, None]) + z[:, :, None], 0, qmax)
    else:
        z = np.full((N, G), float(h), dtype=np.float32)
        q = np.clip(np.rint(Wg / s[:, :, None]), -h, h - 1) + h
    return (q.reshape(N, K).astype(np.uint8), z.astype(np.uint8), s16)


def group_gram(X16, inv_s, group=GROUP, token_chunk=4096):
    """``H_g = X~_g^T X~_g`` for every group g of input channels (fp64
    [G, group, group]), with ``x~ = fp32(x) * inv_s`` as in the layer."""
    X16 = np.asarray(X16, dtype=np.float16)
    T, K = X16.shape
    G = K // group
    H = np.zeros((G, group, group), dtype=np.float64)
    for t0 in range(0, T, token_chunk):
        xt = scaled_activations(X16[t0:t0 + token_chunk], inv_s).astype(np.float64)
        for g in range(G):
            xg = xt[:, g * group:(g + 1) * group]
            H[g] += xg.T @ xg
    return H


def clip_search(X16, W16, s_c, inv_s, n_clip=20, group=GROUP, w_bit=W_BIT, zero_point=True):
    """Per-group clipping ratio by the group's output error (see the READING
    above).  Returns ``(ratio_idx uint8 [N, G], err fp64 [N, G, n_clip])``."""
    W16 = np.asarray(W16, dtype=np.float16)
    N, K = W16.shape
    G = K // group
    H = group_gram(X16, inv_s, group)
    Wp = W16.astype(np.float32)
    if s_c is not None:
        Wp = (Wp * np.asarray(s_c, dtype=np.float32)[None, :]).astype(np.float32)
    Wp = Wp.reshape(N, G, group).astype(np.float64)
    err = np.empty((N, G, n_clip), dtype=np.float64)
    for i in range(n_clip):
        idx = np.full((N, G), i, dtype=np.int64)
        q, z, s16 = quantize_clipped(W16, s_c, idx, n_clip, group, w_bit, zero_point)
        wq = ((q.reshape(N, G, group).astype(np.float64) - z[:, :, None]) *
              s16.astype(np.float64)[:, :, None])
        d = wq - Wp
        err[:, :, i] = np.einsum("ngi,gij,ngj->ng", d, H, d)
    return np.argmin(err, axis=2).astype(np.uint8), err

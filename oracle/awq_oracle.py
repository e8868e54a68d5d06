"""Plain CPU oracle for the AWQ W4A16 / W4A8 quantized linear layer.

TEST INFRASTRUCTURE ONLY: used by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py``; never by the product path.

Sources (web pages, cited by title and section):

* "Speed up AWQ 2.5x with updated kernel" (vLLM pull request), casper-hansen's
  list of format differences: the older ("GEMM") AWQ format packs eight 4-bit
  values per int32 with the order map [0, 2, 4, 6, 1, 3, 5, 7]; zeros are
  packed the same way.  The dispatch snippet on the same page names the
  operands of the kernels: inputs, qweight, scales, qzeros, group_size
  (and split_k_iters for the M > 8 kernel).
* "Marlin symmetric quantization and inference" (AutoAWQ pull request),
  perplexity section: the symmetric variant has no zero points.
* "Support W4A8 quantization for vllm" (vLLM pull request #5218):
  the dynamic per-token activation quantization in brisker's consistency
  script (absmax over the row divided by 127, round, clamp to [-128, 127]);
  HandH1998's answer on per-channel dequantization (int4 to int8 by a left
  shift of 4, the channel scale applied on the output); alexm's review note
  that the reduction works on int32 elements.

Readings taken where the pages are silent (each one is pinned by a test in
``tests/test_oracle_pins.py``):

* order map direction: nibble slot ``i`` (bits 4i..4i+3) of packed word ``c``
  holds logical column ``8c + AWQ_ORDER[i]``;
* dequantization: ``W = fp16_RN((q - z) * s)``, one rounding, subtract first;
  symmetric W4A16 uses z = 8;
* the W4A16 product is reported unrounded in float64 (``linear_f64``) and,
  as the fp32-accumulated variant, in float32 with k ascending
  (``linear_f32acc``); the fp16 output is one RN of the accumulated value;
* W4A8 activation scale: fp16-rounded ``absmax / 127`` widened to fp32 (the
  consistency script divides an fp16 absmax by 127 before converting to
  float); a zero row gets scale 0 and codes 0;
* W4A8 weights: signed int4 q in [-8, 7] stored with the same packing as
  ``u = q + 8``; the int32 accumulator is exact; the output is
  ``fp16_RN((fp32(acc) * s_tok) * fp32(s_ch))``.
"""

from __future__ import annotations

import numpy as np

# Older-format AWQ order map ("Speed up AWQ 2.5x with updated kernel",
# casper-hansen's list of format differences).
AWQ_ORDER = (0, 2, 4, 6, 1, 3, 5, 7)
# The new format's order map (same list): nibble slot i holds column 8c + i.
AWQ_ORDER_NEW = (0, 1, 2, 3, 4, 5, 6, 7)


def unpack(packed: np.ndarray, order=AWQ_ORDER) -> np.ndarray:
    """Unpack an AWQ-packed int32 array [R, C] to 4-bit codes uint8 [R, 8C].

    Nibble slot i of word c holds logical column 8c + order[i] (the older
    format's map by default; ``AWQ_ORDER_NEW`` for the new format's).
    Pins: hand-worked words (golden file), pack/unpack round trip.
    """
    words = np.ascontiguousarray(packed).view(np.uint32)
    rows, cols = words.shape
    out = np.empty((rows, 8 * cols), dtype=np.uint8)
    for slot, col in enumerate(order):
        nib = (words >> np.uint32(4 * slot)) & np.uint32(0xF)
        out[:, col::8] = nib.astype(np.uint8)
    return out


def pack(q: np.ndarray, order=AWQ_ORDER) -> np.ndarray:
    """Pack 4-bit codes uint8 [R, N] (N % 8 == 0) into AWQ int32 words [R, N/8].

    Codes above 15 are clamped to 15 (the W4A8 page reports a packer bug from
    a missing clamp; clamping is the defined behaviour here).  ``order`` as for
    ``unpack``.
    Pins: hand-worked words (golden file), round trip with ``unpack``.
    """
    q = np.asarray(q)
    if q.ndim != 2 or q.shape[1] % 8 != 0:
        raise ValueError("pack expects a 2-D array whose column count is a multiple of 8")
    codes = np.minimum(q.astype(np.uint32), np.uint32(15))
    rows, n = codes.shape
    words = np.zeros((rows, n // 8), dtype=np.uint32)
    for slot, col in enumerate(order):
        words |= codes[:, col::8] << np.uint32(4 * slot)
    return words.view(np.int32)


def dequant(qweight: np.ndarray, qzeros: np.ndarray | None, scales: np.ndarray,
            group_size: int) -> np.ndarray:
    """Group-wise dequantization W[k, n] = fp16_RN((q[k, n] - z[k // g, n]) * s[k // g, n]).

    qweight int32 [K, N/8], qzeros int32 [K/g, N/8] or None (symmetric, z = 8),
    scales fp16 [K/g, N].  Returns fp16 [K, N].

    The product (q - z) * s is exact in float64 (a 5-bit integer times an
    11-bit significand), so the single float64 -> float16 conversion is the
    one correctly rounded step.  Pins: hand-worked values (golden file) and an
    exhaustive (q, z) x scale sweep against exact rational rounding.
    """
    q = unpack(qweight).astype(np.int64)
    k_dim, n_dim = q.shape
    g = int(group_size)
    if g <= 0 or k_dim % g != 0:
        raise ValueError("group_size must divide K")
    n_groups = k_dim // g
    if scales.shape != (n_groups, n_dim):
        raise ValueError("scales must have shape [K/group_size, N]")
    if qzeros is None:
        z = np.full((n_groups, n_dim), 8, dtype=np.int64)
    else:
        z = unpack(qzeros).astype(np.int64)
        if z.shape != (n_groups, n_dim):
            raise ValueError("qzeros must have shape [K/group_size, N/8]")
    group_of_row = np.arange(k_dim) // g
    diff = (q - z[group_of_row, :]).astype(np.float64)
    s = scales.astype(np.float64)[group_of_row, :]
    return (diff * s).astype(np.float16)


def linear_f64(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y[m, n] = sum_k x[m, k] * W[k, n] in float64 (products of two fp16 are exact).

    Pin: brute force with exact rationals at K = 8 (tests).
    """
    return x.astype(np.float64) @ w.astype(np.float64)


def linear_f32acc(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """The same sum accumulated in float32, k ascending (slow; small shapes only).

    Every product of two fp16 values is exact in float32, so only the
    accumulation rounds.  Pin: within K * 2^-24 * sum|x*W| of the exact value.
    """
    x32 = x.astype(np.float32)
    w32 = w.astype(np.float32)
    acc = np.zeros((x.shape[0], w.shape[1]), dtype=np.float32)
    for k in range(x.shape[1]):
        acc += x32[:, k:k + 1] * w32[k:k + 1, :]
    return acc


def awq_linear(x: np.ndarray, qweight: np.ndarray, qzeros: np.ndarray | None,
               scales: np.ndarray, group_size: int) -> np.ndarray:
    """The W4A16 layer: dequantize, then the float64 product (unrounded)."""
    return linear_f64(x, dequant(qweight, qzeros, scales, group_size))


def quant_act(x: np.ndarray):
    """Per-token dynamic int8 quantization of fp16 activations [M, K].

    s[m] = fp32(fp16_RN(fp32(absmax_k |x[m, k]|) / 127)),
    xq[m, k] = clamp(rint(fp32(x[m, k]) / s[m]), -128, 127)   (IEEE fp32 division,
    round half to even).  A row of zeros gets s = 0 and xq = 0.
    Returns (xq int8 [M, K], s float32 [M]).
    Pins: the hand examples in the golden file; |xq| <= 127 with the row's
    absmax element at +-127; zero rows.
    """
    x16 = np.asarray(x, dtype=np.float16)
    absmax = np.abs(x16).max(axis=1).astype(np.float32)
    s = (absmax / np.float32(127.0)).astype(np.float16).astype(np.float32)
    xq = np.zeros(x16.shape, dtype=np.int8)
    nz = s > 0
    if np.any(nz):
        ratio = x16[nz].astype(np.float32) / s[nz, None]
        xq[nz] = np.clip(np.rint(ratio), -128, 127).astype(np.int8)
    return xq, s


def w4a8_accumulate(xq: np.ndarray, wq_packed: np.ndarray) -> np.ndarray:
    """Exact integer accumulator acc[m, n] = sum_k xq[m, k] * (u[k, n] - 8), int64.

    wq_packed holds u = q + 8 in the AWQ packing.  Pin: brute-force integer
    sums on tiny inputs; the result must fit in int32.
    """
    q = unpack(wq_packed).astype(np.int64) - 8
    acc = xq.astype(np.int64) @ q
    if acc.size and (acc.max() > np.iinfo(np.int32).max or acc.min() < np.iinfo(np.int32).min):
        raise OverflowError("W4A8 accumulator does not fit in int32")
    return acc


def w4a8_linear(xq: np.ndarray, s_tok: np.ndarray, wq_packed: np.ndarray,
                s_ch: np.ndarray):
    """W4A8 output y = fp16_RN((fp32(acc) * s_tok[m]) * fp32(s_ch[n])).

    Returns (y fp16 [M, N], acc int64 [M, N]).
    """
    acc = w4a8_accumulate(xq, wq_packed)
    y32 = (acc.astype(np.float32) * np.asarray(s_tok, dtype=np.float32)[:, None])
    y32 = y32 * np.asarray(s_ch, dtype=np.float16).astype(np.float32)[None, :]
    return y32.astype(np.float16), acc


# ---------------------------------------------------------------- bfloat16
# "Support W4A8 quantization for vllm": brisker asks for bf16 because many
# models are trained in bf16; HandH1998 answers that bf16 is not supported
# there.  The bf16 variant of the W4A16 layer takes bf16 activations and
# scales and gives bf16 outputs; numpy has no bf16 type, so bf16 values
# travel here as their uint16 bit patterns (the upper half of an IEEE
# binary32 with the same sign and exponent).

def bf16_to_float(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> the exact values as float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16, to nearest with ties to even; returns uint16 bit patterns.

    bf16 keeps the upper 16 bits of a binary32.  Rounding to nearest adds
    half of the dropped part's weight (0x7FFF) plus the kept part's lowest
    bit (which turns an exact tie towards the even neighbour), then drops
    the lower 16 bits.  Finite inputs only.  Pins: hand-worked values and a
    brute-force nearest-neighbour search over exact rationals (tests).
    """
    f = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    if not np.all(np.isfinite(f)):
        raise ValueError("bf16_round takes finite values")
    bits = f.view(np.uint32).astype(np.uint64)
    keep_lsb = (bits >> np.uint64(16)) & np.uint64(1)
    return ((bits + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)).astype(np.uint16)


def dequant_bf16(qweight: np.ndarray, qzeros: np.ndarray | None, scales_bf16: np.ndarray,
                 group_size: int) -> np.ndarray:
    """W[k, n] = bf16_RN((q[k, n] - z[k // g, n]) * s[k // g, n]) with bf16 scales; bf16 bits [K, N].

    The product of a 5-bit integer and an 8-bit significand is exact in
    float32, so one bf16 rounding of it is the one rounding step.
    """
    q = unpack(qweight).astype(np.int64)
    k_dim, n_dim = q.shape
    g = int(group_size)
    if g <= 0 or k_dim % g != 0:
        raise ValueError("group_size must divide K")
    n_groups = k_dim // g
    if scales_bf16.shape != (n_groups, n_dim):
        raise ValueError("scales must have shape [K/group_size, N]")
    z = np.full((n_groups, n_dim), 8, dtype=np.int64) if qzeros is None else unpack(qzeros).astype(np.int64)
    group_of_row = np.arange(k_dim) // g
    prod = (q - z[group_of_row, :]).astype(np.float64) * bf16_to_float(scales_bf16)[group_of_row, :]
    return bf16_round(prod.astype(np.float32))


def awq_linear_bf16(x_bf16: np.ndarray, qweight: np.ndarray, qzeros: np.ndarray | None,
                    scales_bf16: np.ndarray, group_size: int) -> np.ndarray:
    """The bf16 W4A16 layer: bf16 dequantization, then the float64 product (unrounded).

    Every product of two bf16 values is exact in float64.
    """
    w = bf16_to_float(dequant_bf16(qweight, qzeros, scales_bf16, group_size))
    return bf16_to_float(x_bf16) @ w


# ---------------------------------------------------------------- W4A8 with per-group weight scales
# "Support W4A8 quantization for vllm": HandH1998 says the per-channel kernel
# only uses the channel scale fragment, while per-group weight quantization
# needs both the group and the channel scale; the per-channel path turns an
# int4 weight into an int8 by a shift of 4 (a factor 16) with the channel
# scale on the output; the global reduction works on int32; the GEMM takes
# s1 (per token), s2 and s3.  Reading: s3 is the per-group factor that turns
# an int4 weight into an int8 one, an integer in [1, 16] (16 on every group
# reproduces the per-channel kernel's shift), stored as fp16 [K/g, N]; the
# accumulator stays an exact integer and s2 (per channel) is applied on the
# output exactly like the per-channel scale.

def w4a8_group_accumulate(xq: np.ndarray, wq_packed: np.ndarray, s3: np.ndarray,
                          group_size: int) -> np.ndarray:
    """acc[m, n] = sum_k xq[m, k] * ((u[k, n] - 8) * s3[k // g, n]), exact int64.

    s3 must hold integers in [1, 16] (fp16 storage), so every weight
    (u - 8) * s3 lies in [-128, 112], an int8.  Pins: brute-force integer sums
    on tiny inputs; s3 = 16 everywhere equals 16 times the per-channel
    accumulator.
    """
    s3f = np.asarray(s3, dtype=np.float16).astype(np.float64)
    if np.any(s3f != np.round(s3f)) or np.any(s3f < 1) or np.any(s3f > 16):
        raise ValueError("s3 must hold integers in [1, 16]")
    q = unpack(wq_packed).astype(np.int64) - 8
    k_dim, n_dim = q.shape
    g = int(group_size)
    if g <= 0 or k_dim % g != 0 or s3f.shape != (k_dim // g, n_dim):
        raise ValueError("s3 must have shape [K/group_size, N] with group_size dividing K")
    w8 = q * s3f.astype(np.int64)[np.arange(k_dim) // g, :]
    acc = xq.astype(np.int64) @ w8
    if acc.size and (acc.max() > np.iinfo(np.int32).max or acc.min() < np.iinfo(np.int32).min):
        raise OverflowError("W4A8 accumulator does not fit in int32")
    return acc


def w4a8_group_linear(xq: np.ndarray, s_tok: np.ndarray, wq_packed: np.ndarray, s3: np.ndarray,
                      s2: np.ndarray, group_size: int):
    """Per-group W4A8 output y = fp16_RN((fp32(acc) * s_tok[m]) * fp32(s2[n])), acc from
    ``w4a8_group_accumulate`` (the same epilogue as ``w4a8_linear``, s2 in place of s_ch).

    Returns (y fp16 [M, N], acc int64 [M, N]).
    """
    acc = w4a8_group_accumulate(xq, wq_packed, s3, group_size)
    y32 = (acc.astype(np.float32) * np.asarray(s_tok, dtype=np.float32)[:, None])
    y32 = y32 * np.asarray(s2, dtype=np.float16).astype(np.float32)[None, :]
    return y32.astype(np.float16), acc


# ---------------------------------------------------------------- decode prepack (a private layout)
# "Support W4A8 quantization for vllm": the QQQ kernel shuffles the eight int4
# weights of each int32 offline so that every thread of a warp fetches the
# weights it needs.  The decode GEMV of this library takes an offline-prepared
# copy of an AWQ layer in the layout restated below; the layout changes where
# each code, zero point and scale sits, never its value.
PREPACK_TILE_COLS = 256   # output columns per tile
PREPACK_GROUP = 128       # rows per unit (one quantization group)
PREPACK_UNIT_BYTES = PREPACK_GROUP * PREPACK_TILE_COLS // 2 + PREPACK_TILE_COLS // 2 + 2 * PREPACK_TILE_COLS


def prepack_gemv(qweight: np.ndarray, qzeros: np.ndarray | None, scales: np.ndarray) -> np.ndarray:
    """Prepared decode-GEMV copy of an AWQ layer (group size 128); returns uint8 bytes.

    Units (tile T of 256 columns, group G of 128 rows) follow each other in the
    order T-major, G-minor; each unit is 17024 bytes:
      * 16384 bytes of codes: uint32 words [w 4][i 8][l 32][b 4].  Word
        (w, i, l, b) with g = l // 4, t = l % 4, columns ce = 256 T + 64 w + 8 g + 2 b
        and co = ce + 1, rows k = 128 G + 16 i + (2t, 2t+1, 2t+8, 2t+9) holds, from
        the lowest nibble up: q[2t, ce], q[2t, co], q[2t+8, ce], q[2t+8, co],
        q[2t+1, ce], q[2t+1, co], q[2t+9, ce], q[2t+9, co];
      * 128 bytes of zero points: uint32 words [w 4][g 8]; nibble c of word (w, g)
        is z of column 256 T + 64 w + 8 g + c (8 when ``qzeros`` is None);
      * 512 bytes of scales: fp16 [w 4][g 8][c 8], the scale of the same column.
    Columns at or beyond N get code 0, zero point 0 and scale 0.
    Pins: every code, zero point and scale found again by decoding the layout
    back (tests); the layout's defining cases worked by hand.
    """
    q = unpack(qweight)
    k_dim, n_dim = q.shape
    if k_dim % PREPACK_GROUP:
        raise ValueError("K must be a multiple of 128")
    groups = k_dim // PREPACK_GROUP
    tiles = -(-n_dim // PREPACK_TILE_COLS)
    n_pad = tiles * PREPACK_TILE_COLS
    qp = np.zeros((k_dim, n_pad), dtype=np.uint32)
    qp[:, :n_dim] = q
    zp = np.zeros((groups, n_pad), dtype=np.uint32)
    zp[:, :n_dim] = 8 if qzeros is None else unpack(qzeros)
    sp = np.zeros((groups, n_pad), dtype=np.float16)
    sp[:, :n_dim] = scales
    out = np.zeros((tiles, groups, PREPACK_UNIT_BYTES), dtype=np.uint8)
    # code words: index arrays over (T, G, w, i, l, b)
    T, G, w, i, l, b = np.meshgrid(np.arange(tiles), np.arange(groups), np.arange(4), np.arange(8),
                                   np.arange(32), np.arange(4), indexing="ij")
    g, t = l // 4, l % 4
    ce = 256 * T + 64 * w + 8 * g + 2 * b
    co = ce + 1
    k0 = 128 * G + 16 * i + 2 * t
    nibbles = (qp[k0, ce], qp[k0, co], qp[k0 + 8, ce], qp[k0 + 8, co],
               qp[k0 + 1, ce], qp[k0 + 1, co], qp[k0 + 9, ce], qp[k0 + 9, co])
    words = np.zeros(T.shape, dtype=np.uint32)
    for pos, nib in enumerate(nibbles):
        words |= nib << np.uint32(4 * pos)
    out[:, :, :16384] = words.reshape(tiles, groups, -1).view(np.uint8)
    # zero-point words and scale vectors: [T][G][w][g][c]
    zsel = zp.reshape(groups, tiles, 4, 8, 8).transpose(1, 0, 2, 3, 4)
    zwords = np.zeros((tiles, groups, 4, 8), dtype=np.uint32)
    for c in range(8):
        zwords |= zsel[..., c] << np.uint32(4 * c)
    out[:, :, 16384:16512] = zwords.reshape(tiles, groups, -1).view(np.uint8)
    ssel = sp.reshape(groups, tiles, 4, 8, 8).transpose(1, 0, 2, 3, 4)
    out[:, :, 16512:] = np.ascontiguousarray(ssel).reshape(tiles, groups, -1).view(np.uint8)
    return out.reshape(-1)

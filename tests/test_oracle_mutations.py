"""Planted mistakes in the oracle (on the CPU) must each fail at least one pin.

Each mutant replaces one oracle function with a plausible wrong variant for the
duration of the named pin tests; at least one of them must then fail.  This
shows that the pins in ``test_oracle_pins.py`` constrain the oracle rather than
restate it.
"""

import numpy as np
import pytest

import oracle
from oracle import awq_oracle as O
from tests import test_oracle_pins as pins


def _unpack_inverse_map(packed):
    # wrong direction of the order map
    words = np.ascontiguousarray(packed).view(np.uint32)
    rows, cols = words.shape
    out = np.empty((rows, 8 * cols), dtype=np.uint8)
    for col, slot in enumerate(O.AWQ_ORDER):
        out[:, col::8] = ((words >> np.uint32(4 * slot)) & np.uint32(0xF)).astype(np.uint8)
    return out


def _pack_no_clamp(q):
    codes = np.asarray(q).astype(np.uint32)
    rows, n = codes.shape
    words = np.zeros((rows, n // 8), dtype=np.uint32)
    for slot, col in enumerate(O.AWQ_ORDER):
        words |= codes[:, col::8] << np.uint32(4 * slot)
    return words.view(np.int32)


def _dequant_factory(sign=1, group_mod=False, flip_cols=False, zero=8):
    def dequant(qweight, qzeros, scales, group_size):
        q = O.unpack(qweight).astype(np.int64)
        k_dim, n_dim = q.shape
        g = int(group_size)
        ng = k_dim // g
        z = np.full((ng, n_dim), zero, np.int64) if qzeros is None else O.unpack(qzeros).astype(np.int64)
        gi = (np.arange(k_dim) % ng) if group_mod else (np.arange(k_dim) // g)
        s = scales.astype(np.float64)
        if flip_cols:
            s = s[:, ::-1]
        return (sign * (q - z[gi]).astype(np.float64) * s[gi]).astype(np.float16)
    return dequant


def _linear_transposed(x, w):
    return (w.astype(np.float64).T @ x.astype(np.float64).T).T[:, ::-1]


def _linear_f32acc_fp16_accum(x, w):
    acc = np.zeros((x.shape[0], w.shape[1]), dtype=np.float16)
    for k in range(x.shape[1]):
        acc += x[:, k:k + 1] * w[k:k + 1, :]
    return acc.astype(np.float32)


def _quant_act_fp32_scale(x):
    x16 = np.asarray(x, dtype=np.float16)
    s = np.abs(x16).max(axis=1).astype(np.float32) / np.float32(127)
    xq = np.zeros(x16.shape, np.int8)
    nz = s > 0
    xq[nz] = np.clip(np.rint(x16[nz].astype(np.float32) / s[nz, None]), -128, 127).astype(np.int8)
    return xq, s


def _quant_act_half_up(x):
    x16 = np.asarray(x, dtype=np.float16)
    s = (np.abs(x16).max(axis=1).astype(np.float32) / np.float32(127)).astype(np.float16).astype(np.float32)
    xq = np.zeros(x16.shape, np.int8)
    nz = s > 0
    xq[nz] = np.clip(np.floor(x16[nz].astype(np.float32) / s[nz, None] + 0.5), -128, 127).astype(np.int8)
    return xq, s


def _w4a8_acc_offset7(xq, wq):
    return xq.astype(np.int64) @ (O.unpack(wq).astype(np.int64) - 7)


def _w4a8_linear_factory(kind):
    # wrong W4A8 epilogues: the token scale dropped, the scale product taken first, an fp16 intermediate
    # after the token scale, and the whole chain in float64 (no fp32 rounding of acc or the products)
    def w4a8_linear(xq, s_tok, wq_packed, s_ch):
        acc = O.w4a8_accumulate(xq, wq_packed)
        st = np.asarray(s_tok, dtype=np.float32)[:, None]
        sc = np.asarray(s_ch, dtype=np.float16).astype(np.float32)[None, :]
        a32 = acc.astype(np.float32)
        if kind == "drop_tok":
            y = a32 * sc
        elif kind == "product_first":
            y = a32 * (st * sc)
        elif kind == "fp16_intermediate":
            y = (a32 * st).astype(np.float16).astype(np.float32) * sc
        else:
            y = acc.astype(np.float64) * st.astype(np.float64) * sc.astype(np.float64)
        return y.astype(np.float16), acc
    return w4a8_linear


def _bf16_round_truncate(v):
    f = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _bf16_round_ties_away(v):
    f = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    return ((f.view(np.uint32).astype(np.uint64) + np.uint64(0x8000)) >> np.uint64(16)).astype(np.uint16)


def _dequant_bf16_zero7(qweight, qzeros, scales_bf16, group_size):
    q = O.unpack(qweight).astype(np.int64)
    k_dim, n_dim = q.shape
    g = int(group_size)
    z = np.full((k_dim // g, n_dim), 7, np.int64) if qzeros is None else O.unpack(qzeros).astype(np.int64)
    gi = np.arange(k_dim) // g
    prod = (q - z[gi]).astype(np.float64) * O.bf16_to_float(scales_bf16)[gi]
    return O.bf16_round(prod.astype(np.float32))


def _group_acc_factory(kind):
    def acc_fn(xq, wq_packed, s3, group_size):
        q = O.unpack(wq_packed).astype(np.int64) - 8
        k_dim, n_dim = q.shape
        g = int(group_size)
        s3i = np.asarray(s3, dtype=np.float16).astype(np.int64)
        gi = (np.arange(k_dim) % (k_dim // g)) if kind == "group_mod" else (np.arange(k_dim) // g)
        if kind == "offset7":
            q = q + 1
        return xq.astype(np.int64) @ (q * s3i[gi, :])
    return acc_fn


def _prepack_swapped_columns(qweight, qzeros, scales):
    # even and odd columns of each block swapped
    q = O.unpack(qweight)
    q2 = q.reshape(q.shape[0], -1, 2)[:, :, ::-1].reshape(q.shape)
    return _ORIGINAL_PREPACK(O.pack(q2), qzeros, scales)


_ORIGINAL_PREPACK = O.prepack_gemv

MUTANTS = [
    ("unpack", _unpack_inverse_map, ["test_unpack_pack_golden"]),
    ("pack", _pack_no_clamp, ["test_pack_clamps_codes_above_15"]),
    ("dequant", _dequant_factory(sign=-1), ["test_dequant_golden"]),
    ("dequant", _dequant_factory(group_mod=True), ["test_dequant_group_index_closed_form"]),
    ("dequant", _dequant_factory(flip_cols=True), ["test_dequant_per_column_scale_and_zero_not_transposed"]),
    ("dequant", _dequant_factory(zero=7), ["test_dequant_symmetric_uses_zero_eight"]),
    ("linear_f64", _linear_transposed, ["test_linear_bruteforce_exact_rationals"]),
    ("linear_f32acc", _linear_f32acc_fp16_accum, ["test_linear_bruteforce_exact_rationals"]),
    ("quant_act", _quant_act_fp32_scale, ["test_quant_act_golden"]),
    ("quant_act", _quant_act_half_up, ["test_quant_act_golden"]),
    ("w4a8_accumulate", _w4a8_acc_offset7, ["test_w4a8_accumulate_bruteforce"]),
    ("w4a8_linear", _w4a8_linear_factory("drop_tok"), ["test_w4a8_epilogue_golden"]),
    ("w4a8_linear", _w4a8_linear_factory("product_first"), ["test_w4a8_epilogue_golden"]),
    ("w4a8_linear", _w4a8_linear_factory("fp16_intermediate"), ["test_w4a8_epilogue_golden"]),
    ("w4a8_linear", _w4a8_linear_factory("float64"), ["test_w4a8_epilogue_golden"]),
    ("bf16_round", _bf16_round_truncate, ["test_bf16_golden", "test_bf16_round_is_the_nearest_bf16"]),
    ("bf16_round", _bf16_round_ties_away, ["test_bf16_golden", "test_bf16_round_is_the_nearest_bf16"]),
    ("dequant_bf16", _dequant_bf16_zero7, ["test_dequant_bf16_symmetric_and_group_index"]),
    ("w4a8_group_accumulate", _group_acc_factory("group_mod"), ["test_w4a8_group_accumulate_bruteforce"]),
    ("w4a8_group_accumulate", _group_acc_factory("offset7"), ["test_w4a8_group_accumulate_bruteforce",
                                                               "test_w4a8_group_factor_16_is_the_per_channel_kernel"]),
    ("prepack_gemv", _prepack_swapped_columns, ["test_prepack_words_for_row_and_column_patterns"]),
]


@pytest.mark.parametrize("name,mutant,pin_names", MUTANTS,
                         ids=[f"{m[0]}-{i}" for i, m in enumerate(MUTANTS)])
def test_planted_mistake_fails_a_pin(monkeypatch, golden_dir, name, mutant, pin_names):
    monkeypatch.setattr(O, name, mutant)
    monkeypatch.setattr(oracle, name, mutant)
    failed = False
    for pin in pin_names:
        fn = getattr(pins, pin)
        try:
            if "golden_dir" in fn.__code__.co_varnames[:fn.__code__.co_argcount]:
                fn(golden_dir)
            else:
                fn()
        except Exception:
            failed = True
    assert failed, f"mutant of {name} passed {pin_names}"

"""CPU oracle for the AWQ W4A16 / W4A8 quantized linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` use it.  It shares no code with
the CUDA library (``bit_weight_only_awq_gb300/csrc``) and imports nothing from
it.

Every function here is a plain, slow, readable restatement of what the
quantized linear layer computes; see ``awq_oracle`` for the per-function
citations and for which pins (``tests/test_oracle_pins.py``) hold each
function to something other than itself.
"""

from .awq_oracle import (  # noqa: F401
    AWQ_ORDER,
    AWQ_ORDER_NEW,
    unpack,
    pack,
    dequant,
    linear_f64,
    linear_f32acc,
    awq_linear,
    quant_act,
    w4a8_accumulate,
    w4a8_linear,
    bf16_to_float,
    bf16_round,
    dequant_bf16,
    awq_linear_bf16,
    w4a8_group_accumulate,
    w4a8_group_linear,
    PREPACK_UNIT_BYTES,
    prepack_gemv,
)

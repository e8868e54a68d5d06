"""GB300-native AWQ W4A16 / W4A8 weight-only quantized linear layer.

The compute path is the C-ABI library ``libawq.so`` (hand-written sm_103a
CUDA, declared in ``include/awq.h``); ``bit_weight_only_awq_gb300.awq`` is a
thin ctypes binding over it with the same entry-point names.  Importing the
package does not load the library; importing ``bit_weight_only_awq_gb300.awq``
does, and fails loudly if the library has not been built.
"""

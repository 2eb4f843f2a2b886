"""GB300-native exact attention (FlashAttention-2-style online softmax), fwd and bwd.

The compute path is the CUDA library ``libfa.so`` built from ``csrc/`` for sm_103a;
``exact_attention_38_gb300.fa`` is its thin ctypes binding.  Importing this
package does not load the library; importing ``.fa`` does, and fails loudly if
the library is missing.
"""

__all__ = ["fa", "inputs"]

"""CPU oracle for the INT4 group-compressed OPT decoder layer -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement of what the hot path computes, written
from the FlexGen pages:

* group-wise asymmetric 4-bit quantisation of weights (groups of 64 along the output
  channel) and of the KV cache (groups of 64 along the hidden dimension), with a
  per-group min ``a`` and max ``b``, values dequantised to FP16 before compute
  (FlexGen review, jaehun.me, section "4-bit 압축은 정수 연산 가속과 같은가", paper §5;
  "论文阅读：FlexGen", blog.gzher.com, §3.4 "4-bit 压缩权重和 KV cache");
* one pre-LN OPT decoder layer applied to a block of sequences, prefill over the
  prompt then decode steps that extend the cache (FlexGen paper explainer,
  "Problem Formulation" and Figure 2; Algorithm 1).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
arm may import this package.  The product path (the CUDA library and its binding)
never imports, links or executes anything here, and this package imports nothing from
the product path: the two share no code.  The only shared module is ``fg_synth``,
which draws seeded inputs and holds none of the method's arithmetic.

Parity status of each function is stated in its docstring.  Everything in
``quant.py`` is pinned (tests/test_oracle_quant.py).  ``layer.py`` is pinned by
brute-force loops on tiny inputs, closed forms and invariants
(tests/test_oracle_layer.py); absolute layer values at full size have no printed
counterpart on the pages and are pinned only through those checks.
"""
from .quant import (quantize_g64, dequant_g64, pack_nibbles, unpack_nibbles,  # noqa: F401
                    group_min_max, ab_pack_u32)
from .layer import (layernorm, relu, causal_attention, decode_attention,  # noqa: F401
                    QuantLayer, KVCache, layer_prefill, layer_decode, run_stack)

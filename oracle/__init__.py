"""CPU oracle for exact causal, segment-masked softmax attention (test infrastructure).

This package is test infrastructure only. The product path (the CUDA library and
its Python binding) never imports, calls or links anything here; only the tests,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` use it.

Source of the definition: "World Model on Million-Length Video And Language With
Blockwise RingAttention" (LWM, arXiv 2402.08268) as summarised on the
charles2530.github.io deep-dive page:
  * section "RingAttention 为什么必要": the attention is exact full attention, with
    no sliding window or sparse approximation, computed block by block;
  * section "模型结构": the model is an autoregressive next-token Transformer, so
    attention is causal;
  * section "Masked sequence packing": several samples share one packed row and an
    attention mask lets each sample attend only to itself.

Everything is computed in float64 with NumPy (BLAS matmul as a primitive step).
"""

from .attention import (  # noqa: F401
    visible_mask,
    attention_forward,
    attention_backward,
    attention_forward_rows,
    attention_backward_rows,
    attention_key_grads,
    forward_row_block,
    backward_row_block,
    credited_pairs,
)
from .rope import (  # noqa: F401
    rope_angles,
    rope_rotate,
    round_bf16,
    attention_forward_rope,
    attention_backward_rope,
)
from .loss_weighting import (  # noqa: F401
    documents,
    token_cross_entropy,
    packed_loss,
)

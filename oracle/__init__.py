"""fp64 CPU oracle for one Qwen3-style decoder layer and the lm-head loss.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it. It shares no code with
the CUDA library (``bwd_qwen3_layer_gb300/csrc``); the only module both sides
use is the seeded input generator ``bwd_qwen3_layer_gb300.synth``, which holds
none of the method's arithmetic.

Sources (public web pages on the subject):

* "From-scratch GPU LLM training" (keilab.pages.dev/ai/gpu-llm and its
  markdown twin keilab.io/ai/gpu-llm/index.md, section "What is built"): the
  six gradient kernels (matrix multiply, RMSNorm, SiLU/SwiGLU, RoPE, softmax
  cross-entropy, scaled-dot-product attention), the layer backward that
  chains them, the lm-head softmax cross-entropy fused with argmax, and the
  layer-streaming forward; gradient clipping in the end-to-end smoke bullet.
* "KYNETRA FOUNDRY" (hyperbridge-deck.pages.dev): the pre-normalisation
  decoder paragraph (RMSNorm -> causal self-attention -> SwiGLU FFN, each in
  a residual), the grouped-query attention paragraph, the rotary position
  paragraph, and the tiled-attention paragraph (tiling is an exact IO
  reordering of plain attention, so the oracle computes plain attention).

Where the pages leave a step open the oracle takes one reading and says so in
the function that implements it (pairing of rotary planes, GQA group
mapping, epsilon placement, loss reduction, argmax tie-break, clip formula).

Every function here is pinned by ``tests/test_oracle_*.py`` against something
other than itself: central finite differences, brute-force loops, closed
forms, invariants and special cases. None is "parity unpinned".
"""

from .qwen3_layer import (  # noqa: F401
    LayerConfig,
    attention_bwd,
    attention_fwd,
    attention_fwd_rows,
    ce_argmax,
    layer_backward,
    layer_forward,
    linear,
    lmhead_ce,
    rmsnorm_bwd,
    rmsnorm_fwd,
    rope_angles,
    rope_bwd,
    rope_fwd,
    silu,
    swiglu_bwd,
    swiglu_fwd,
)
from .stack import stack_fwd_bwd, clip_coefficient  # noqa: F401
from .paged import (  # noqa: F401,E402
    gather,
    layer_forward_paged,
    paged_attention,
    paged_write,
    positions,
    rope_at,
)

"""Float64 CPU oracle of the headwise-chunked causal GQA attention layer, and
of the sequence-tiled MLP and loss around it.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline of ``bench.py`` use it.  It shares no code with the CUDA path and is
never called by it.  Every function cites the passage it follows; see
``attention_layer`` for the readings taken where the pages are silent.
"""
from .attention_layer import (  # noqa: F401
    apply_rope, apply_rope_transpose, causal_attention,
    layer_backward, layer_backward_key_rows, layer_backward_tail, layer_forward, layer_loss, project_kv, rms_norm,
    rms_norm_backward, rope_cos_sin,
)
from .mlp import (  # noqa: F401
    mlp_backward, mlp_forward, mlp_loss, sigmoid, silu, silu_grad,
)
from .loss import (  # noqa: F401
    logsumexp_rows, loss_backward, loss_forward, loss_total,
)

"""CPU float64 oracle for the LoRA block projections -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The CUDA library never calls it, and it shares no code with
the CUDA path: it is plain numpy in float64.

See :mod:`oracle.lora` for what is computed and which passage of the pages each
function follows.
"""

from .lora import (  # noqa: F401
    ACTS, act, act_prime, silu, gelu_tanh, gelu_erf, lora_linear, lora_linear_grad,
    mlp_forward, mlp_backward, mlp_backward_per_example, qkvo_forward, qkvo_backward, linear_t,
    rope_tables, apply_rope, apply_rope_transpose,
)

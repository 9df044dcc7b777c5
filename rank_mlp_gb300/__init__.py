"""GB300 (sm_103a) LoRA block projections: the gated MLP (gate/up + SwiGLU or
tanh-GeGLU + down) and the Q/K/V + O projections, forward and backward, behind the
C ABI declared in ``include/lora_gb300.h``.

``rank_mlp_gb300.binding`` is the Python binding (argument marshalling over ctypes;
every step runs in the library's CUDA kernels).  ``rank_mlp_gb300.autograd`` wraps the
same calls as torch.autograd functions (frozen W; gradients for x, A, B).
``rank_mlp_gb300.build`` compiles the library in-tree.
"""

__all__ = ["autograd", "binding", "build"]

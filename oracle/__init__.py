"""CPU oracle for the fused MoE-FFN layer.

Test infrastructure only: the test suite, the smoke check and the benchmark's
CPU-baseline leg may import it; the product path (the CUDA library and its
Python binding) never does, and shares no code with it.
"""
from .moe_ffn import (route, dispatch, combine, silu, swiglu, swiglu_grad,  # noqa: F401
                      expert_forward, expert_backward, forward, backward, shared_expert_forward,
                      token_outputs, expert_weight_grads)

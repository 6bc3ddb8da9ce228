"""fp64 CPU oracle for the fused attention forward.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke entry point and by the
benchmark's CPU-baseline leg, never by the library. It shares no code with the
CUDA path. ``attention`` is the two-pass definition; ``online_softmax`` is an
independently written tiled recurrence used to cross-check it on tiny inputs.
``fp8_quant`` holds the e4m3 block quantisation and Hadamard rotation;
``attention_varlen`` the ragged-batch (cumulative offsets) forward;
``attention_backward`` the gradients dQ, dK, dV.
"""
from .attention import attention_forward, attention_head, kv_head, probabilities, scores, softmax_two_pass
from .online_softmax import attention_online
from . import fp8_quant
from .varlen import attention_varlen
from .backward import attention_backward, attention_backward_head

__all__ = ["attention_forward", "attention_head", "kv_head", "probabilities", "scores",
           "softmax_two_pass", "attention_online", "fp8_quant", "attention_varlen",
           "attention_backward", "attention_backward_head"]

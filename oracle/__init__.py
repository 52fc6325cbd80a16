"""Double-precision CPU oracle (test infrastructure only; see ``attention.py``)."""
from .attention import (alibi_bias, allowed, backward, backward_cols, backward_rows, forward, forward_rows, preprocess_D,
                        reference_grads, tensor_bias, varlen_backward, varlen_forward)
from .philox import drop_threshold, keep_mask, philox4x32_10

__all__ = ["alibi_bias", "allowed", "backward", "backward_cols", "backward_rows", "forward", "forward_rows", "preprocess_D",
           "reference_grads", "tensor_bias", "varlen_backward", "varlen_forward",
           "drop_threshold", "keep_mask", "philox4x32_10"]

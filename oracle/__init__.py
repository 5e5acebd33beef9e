"""CPU fp64 oracle for blocked GQA flash attention (test infrastructure only).

Imported only by the tests, by ``__graft_entry__.smoke()`` and by the CPU
baseline / reference legs of ``bench.py``; never by the product path."""
from .attention import (attention_backward, attention_backward_rows,
                        attention_bruteforce, attention_forward,
                        attention_mask, attention_rows, masked_softmax)

__all__ = [
    "attention_backward", "attention_backward_rows", "attention_bruteforce",
    "attention_forward", "attention_mask", "attention_rows", "masked_softmax",
]

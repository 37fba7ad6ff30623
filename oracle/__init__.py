"""fp64 CPU oracle for the online-softmax attention forward and the row (m, l) state.

TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library and its
Python binding) imports, links or runs this package; only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg use it.  It shares
no code with the CUDA path: it receives plain numpy arrays and returns numpy
arrays.

Every function computes the plain definition the pages give, in float64, with no
blocking, fusion or reordering beyond what the definition states:

* ``row_state``          -- per-row (m, l) of the safe softmax
                            ("Softmax 数值稳定性与 IO-Aware Attention：从在线归一化到
                            FlashAttention", §二 2.1 and §三).
* ``softmax_rows``       -- the normalised row softmax, pass three of §三.
* ``attention_forward``  -- standard attention S = scale*Q K^T, P = softmax(S),
                            O = P V, plus LSE = m + ln l (same page, §七; the
                            scale follows "为什么 Flash Attention 算出来的结果和标准
                            注意力有微小差异？有损但值得", section "它没省计算，只是
                            把矩阵拆开再算").
* ``attention_backward`` -- dQ, dK, dV of that function for an upstream dO, by the
                            chain rule (``oracle.backward``; §7.2 of the first page
                            named above says the backward recomputes the scores from
                            kept statistics, §九 9.1 asks for gradient checks).

The online forms in ``oracle.online`` restate the pages' recurrences and are used
only to cross-check the three-pass forms above.  Parity status of every function
is pinned by ``tests/test_oracle_pins.py``; no function here is unpinned.
"""

from .reference import attention_forward, row_state, softmax_rows, visible_mask
from .backward import attention_backward, attention_backward_rows
from .online import (
    online_weighted_sum,
    online_state,
    merge_state,
    tiled_attention_forward,
    combine_partials,
)

__all__ = [
    "attention_forward",
    "attention_backward",
    "attention_backward_rows",
    "row_state",
    "softmax_rows",
    "visible_mask",
    "online_weighted_sum",
    "online_state",
    "merge_state",
    "tiled_attention_forward",
    "combine_partials",
]

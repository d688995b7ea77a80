"""Plain CPU oracle for one tree-verification step of Medusa/Hydra speculative decoding.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may use it.  It shares no code, table or helper with the
CUDA library; the two meet only through the seeded generators of
``spec_workloads`` (which hold none of the method's arithmetic).

Everything here is written for a reader checking it against the pages by eye:
NumPy in float64, no blocking, no fusion, no online softmax.  Each function
cites the passage it follows:

* "Hydra Guide: Sequentially-Dependent Speculative AI" (aifetchly blog), the
  sections on embedding conditioning, candidate tree construction, the tree
  attention matrix and greedy acceptance;
* "Speculative Decoding" (thegustafson.com), the sections on the acceptance
  criterion (including what happens to the caches after it), the correctness
  guarantee and the worked example;
* "Medusa Heads" (ultralytics glossary), the sections on how the heads predict
  and on tree attention and acceptance;
* Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3"
  (SC'11) for the Philox counter-based generator, which the pages do not give.

Parity pins (all in ``tests/test_oracle_*.py``, CPU only): every function is
pinned by something other than itself -- a library routine it should reduce
to, a value printed on the pages, a closed form, or brute force.  No function
here is "parity unpinned".
"""

from .bf16 import bf16_bits_to_f64, f64_to_bf16_bits
from .tree import tree_encode, tree_mask
from .heads import silu, hydra_draft, hydra_draft_heads
from .attention import tree_attention, tree_attention_paged, gather_pages
from .accept import greedy_accept, rejection_accept, typical_accept
from .kv_commit import kv_commit, kv_commit_paged
from .philox import philox4, philox4x32_10, philox_uniform_pair, uniform_from_u32

__all__ = [
    "bf16_bits_to_f64", "f64_to_bf16_bits",
    "tree_encode", "tree_mask",
    "silu", "hydra_draft", "hydra_draft_heads",
    "tree_attention", "tree_attention_paged", "gather_pages",
    "greedy_accept", "rejection_accept", "typical_accept", "kv_commit",
    "philox4", "philox4x32_10", "philox_uniform_pair", "uniform_from_u32",
    "kv_commit_paged",
]

"""fp64 CPU oracle of the verify-and-commit step.

Test infrastructure only: imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference leg.  It shares no code with the
CUDA library and is never on the product path.
"""
from .spec_oracle import *  # noqa: F401,F403
from .spec_oracle import (BOUNDARY_MARGIN, DEFAULT_EPS, FLAG_BAD_INPUT, FLAG_BAD_ROW,  # noqa: F401
                          FLAG_FALLBACK)
from .ngram_oracle import NgramDraft, ngram_draft  # noqa: F401
from .tree_build_oracle import Level, Tree, build_tree, expand_level  # noqa: F401

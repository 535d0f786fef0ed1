"""FP64 CPU oracle for the flow-matching action-decoder hot path.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import anything from here. The GPU
library never calls, links or reads it, and it never imports the GPU library.

Parity pins (see tests/test_oracle_*.py): every function is checked against
closed forms, format definitions, independent library codecs, invariants, or a
brute-force scalar restatement on tiny shapes. Agreement with FlashRT-PAI's or a
trained policy's actual numbers is "parity unpinned": the pages print no layer
values or actions and no trained weights exist here.
"""
from . import codecs, model  # noqa: F401

"""CPU oracle for paged-KV attention — TEST INFRASTRUCTURE.

Plain NumPy float64 definitions of what the library computes, used only by
the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``. The library never imports, links or runs anything here, and
nothing here imports the library.
"""
from .core import (  # noqa: F401
    OracleInputError,
    attend_partial,
    attend_row,
    combine_splits,
    gather_sequence,
    kv_append,
    live_slots,
    pack_tick,
    paged_attention,
    pool_bytes,
)

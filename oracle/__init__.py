"""CPU fp64 oracle of the MoE layer.  Test infrastructure only: imported by
``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``,
never by the library."""

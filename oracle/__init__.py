"""CPU oracle for routed MoE expert-parallel dispatch / combine.

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline leg, never by the library. ``ref`` wraps
the C counter-loop oracle; ``sort_oracle`` is an independent stable-sort
formulation of the dispatch metadata used to pin it.
"""

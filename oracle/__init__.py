"""CPU fp64 oracle of the decode layer and of the pipeline's schedule model.

TEST INFRASTRUCTURE ONLY: imported by the tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``; never by the product path.
"""

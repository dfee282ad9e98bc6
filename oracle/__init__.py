"""fp64 CPU oracle for the Gated DeltaNet token mixer.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it to check and to time against; the
product package never imports it, and it shares no code with the CUDA path.
"""

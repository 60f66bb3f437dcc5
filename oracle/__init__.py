"""CPU oracle for paged KV storage and paged attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check in ``__graft_entry__`` and the
benchmark's CPU-baseline leg (``bench.py`` ``cpu_baseline`` and ``--impl reference``) may
import this package.  The product library never does, and shares no code with it.

* ``kvc_oracle.c`` -- fp64 address rule, slot mapping, store, gathered attention and the
  log-sum-exp merge of split partials (plain C, compiled with gcc, loaded by ctypes).
* ``oracle.py`` -- ctypes marshalling for it (numpy arrays in and out, no arithmetic).
* ``plan.py`` -- Quail's prefix-sharing plan (pure Python).
"""

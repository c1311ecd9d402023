"""CPU oracle (test infrastructure only; see ``nf4_oracle``).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
legs may import this package.  The product never does.
"""

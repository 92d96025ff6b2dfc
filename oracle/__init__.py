"""CPU oracle for row-wise RMSNorm forward/backward, and the correctness gate.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` may import this package. The GPU library and its
Python binding never import it, and it never imports them.

Contents:
  * ``oracle.oracle``: ctypes front end of ``rmsnorm_oracle.c`` (fp64 golden and
    same-dtype fp32-intermediate reference, plus exact number-format helpers).
  * ``oracle.gate``: the golden / reference / target correctness gate and the
    conditioning check of the torchtitan kernel-numerics page.
"""

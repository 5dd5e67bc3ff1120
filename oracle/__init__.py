"""CPU float64 oracle for the DP-SGD private-gradient step (clip + noise).

TEST INFRASTRUCTURE ONLY.  This package is the slow, plain, obviously
correct restatement of what the GPU library computes, used to prove parity.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  The product path (``differentially_private_gb300``
and its CUDA library) never imports, links or calls anything here, and this
package imports nothing from the product path: the two share no code.  The
only thing they share is input bytes produced by the seeded generators in
``synthetic/``.

Modules
-------
``philox``  Philox4x32-10 counter-based generator (Salmon, Moraes, Dror, Shaw,
            "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11) and the
            Box-Muller map from its words to standard normals.
``dpsgd``   per-example gradients, norms, clip factors, clipped sum, noise and
            normalisation of one DP-SGD step, in float64.

Parity status of each function is stated in its module header.
"""

from . import philox, dpsgd  # noqa: F401

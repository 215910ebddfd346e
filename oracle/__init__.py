"""CPU oracle for the chunked gated-delta-rule scan.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library and
its Python binding never import it, and it imports nothing from them.

Contents
--------
``recurrence``  fp64 token-by-token recurrence in C (forward, reverse mode,
                segment summary, merge), loaded with ctypes.
``chunk_form``  fp64 numpy statement of the 64-token chunk algorithm that
                defines the intermediate outputs (cumulative gate, A, w, u,
                v_new, per-chunk entry states) and its reverse mode.
``frame_scan``  fp64 numpy statement of the dense per-token transition scan (right-
                multiply KV and left-multiply Z states, truncation, the
                segment-split correction).
``brute``       exact rational (``fractions.Fraction``) unrolled-product form
                of the recurrence for tiny inputs; the pin for ``recurrence``.
"""
from . import brute, chunk_form, frame_scan, recurrence  # noqa: F401

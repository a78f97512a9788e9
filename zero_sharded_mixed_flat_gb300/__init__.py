"""zero_sharded_mixed_flat_gb300: the sharded mixed-precision optimizer step
(ZeRO stage two over a flat parameter vector) as hand-written CUDA for GB300.

The compute lives in the C-ABI library ``libzg.so`` (sources in ``csrc/``,
declarations in ``include/zg.h``). ``binding`` is a thin ctypes layer over it
that takes torch tensors for device memory and streams. ``synth`` draws the
seeded synthetic inputs and ``accounting`` holds the byte formulas.

Importing this package loads nothing; the library is loaded on first use of
``binding`` and the import fails loudly if it has not been built.
"""

__all__ = ["binding", "synth", "accounting"]

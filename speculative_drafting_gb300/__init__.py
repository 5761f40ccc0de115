"""P-EAGLE parallel-draft step on GB300 (sm_103a).

The step runs in the CUDA library ``libpe.so`` (sources in ``csrc/``, C-ABI in
``include/pe.h``); ``binding`` is a thin ctypes layer over it.  Importing the
package does not load the library; ``binding.load()`` does, and fails loudly
when it has not been built.
"""

__all__ = ["workloads", "binding", "build"]

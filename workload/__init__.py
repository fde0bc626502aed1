"""Seeded synthetic inputs for the FASA decode step.

This module is the only code shared by the oracle side and the CUDA side of
the tests and the benchmark.  It holds no arithmetic of the method (no TIP
score, no selection, no attention): it draws pre-RoPE queries and keys,
values, outlier frequency chunks and dominant-FC tables, and stores the keys
the way a KV cache holds them, i.e. after their rotary encoding at their own
positions.  That key rotation is input preparation and is implemented here on
its own; neither the oracle nor the library imports it.

Two generators produce the same recipe:

* ``synth.py``  -- numpy, host side, for the small cases and the CPU tests.
* ``csrc/synth_gen.cu`` -- a CUDA kernel (built into ``libfasa_synth.so``)
  for the large cases, loaded through ``gpu_gen.py``.

Both draw normals from one counter-based generator, SplitMix64 (Steele, Lea
and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014)
feeding the Box-Muller transform.  Every test compares the library against
the oracle on the *stored bytes* that were actually fed to the GPU, so the
two generators never have to agree bit for bit.
"""

from .configs import CONFIGS, Config, get_config  # noqa: F401

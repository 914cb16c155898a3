"""GB300-native attention hot path of a bounded-generation SLM inference engine.

Three C-ABI entry points (``include/bg_attn.h``) implemented with hand-written
sm_103a CUDA kernels:

  * ``bg_packed_prefill_attn``  packed variable-length causal GQA prefill
  * ``bg_beam_decode_attn``     beam-search decode over a shared prompt K/V
                                plus per-beam suffix K/V
  * ``bg_beam_suffix_reorder``  bit-exact reorder of the per-beam suffix by the
                                beam parent index (with optional append of the
                                step's new token)

``binding`` is a thin ctypes layer over the shared library; importing this
package does not load the library (so CPU-only tooling can import
``workloads``).  The library must be built first (``build.build()``); the
binding raises if it is missing -- there is no CPU fallback.
"""

__all__ = ["binding", "workloads", "build"]

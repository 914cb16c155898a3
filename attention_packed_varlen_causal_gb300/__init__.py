"""GB300-native attention hot path of a bounded-generation SLM inference engine.

C-ABI entry points (``include/bg_attn.h``), all implemented with hand-written
sm_103a CUDA kernels:

  * ``bg_packed_prefill_attn``        packed variable-length causal GQA prefill
    (+ ``bg_packed_prefill_workspace_size``)
  * ``bg_packed_prefill_attn_fp8``    the same with E4M3 Q and K (per-tensor
                                      power-of-two scales) and a bf16 V
  * ``bg_packed_prefill_attn_noalloc``  the prefill for callers that cannot
                                      allocate (fixed scratch in the library)
  * ``bg_packed_last_token_attn``     attention of each sequence's last valid
                                      token only (Prefill-Only last layer)
  * ``bg_beam_decode_attn``           beam-search decode over a shared prompt
                                      K/V plus per-beam suffix K/V
  * ``bg_beam_suffix_reorder``        bit-exact reorder of the per-beam suffix
                                      by the beam parent index (optional append)
  * ``bg_beam_decode_step``           one whole decode step: reorder + append
                                      of the suffix and the decode attention
  * ``bg_beam_select``                beam candidate selection of one step
    (+ ``bg_beam_select_workspace_size``)
  * ``bg_selftest_wait_timeout``      diagnostic of the bounded-wait failure path
  * ``bg_status_string``

``binding`` is a thin ctypes layer over the shared library; importing this
package does not load the library (so CPU-only tooling can import
``workloads``).  The library must be built first (``build.build()``); the
binding raises if it is missing -- there is no CPU fallback.
"""

__all__ = ["binding", "workloads", "build"]

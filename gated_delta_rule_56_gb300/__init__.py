"""Kimi Delta Attention (KDA) prefill and decode for GB300 (sm_103a).

The computation lives in libkda.so (hand-written CUDA, C ABI in include/kda.h); this
package is its thin Python binding:

* ``prefill(q, k, v, g, beta, cu_seqlens=None, initial_state=None)`` -> (o, final_state)
* ``decode_step(q, k, v, g, beta, state)`` -> o   (state updated in place)
* ``backward(q, k, v, g, beta, d_o, ...)`` -> dict of gradients (fp32)
* ``prefill_split_plan(B, T, H, sm_count)`` -> how a call of these sizes is split along the
  sequence (segments, rows per segment, workspace bytes); host arithmetic only
* ``check_status()`` -> raises ``KDAError`` if a kernel flagged a device-side error
* ``selftest_wait_timeout(limit_ns)`` -> queues the bounded-wait self-test (a time-out that the
  next ``check_status()`` reports)

Build the library with ``gated_delta_rule_56_gb300.build.build()``.
"""

from ._lib import (KDAError, backward, check_status, declared_symbols, decode_step, last_error, library_path,
                   load, prefill, prefill_split_plan, selftest_wait_timeout, status_string, version)

__all__ = ["KDAError", "backward", "check_status", "declared_symbols", "decode_step", "last_error", "library_path",
           "load", "prefill", "prefill_split_plan", "selftest_wait_timeout", "status_string", "version"]

"""KDA bounded-gate linear attention on GB300 (sm_103a).

Four calls, backed by libkda's CUDA kernels (``include/kda.h``):

* :func:`chunk_prefill` -- chunked varlen prefill with a pooled fp32 state;
* :func:`recurrent_verify` -- speculative-decode verify writing every per-step state;
* :func:`commit_accepted` -- accept/commit: the state after the last accepted draft token back into the pool;
* :func:`spec_step` -- one speculative-decoding step: prefill segment and verify segment in one call, their
  outputs written straight into the layer's output rows by index.

Optional parts of a layer step, taken by the calls above:

* :class:`OutputNorm` -- sigmoid-gated RMSNorm of every output row (``norm=``);
* :class:`ShortConv` -- short causal convolutions of q, k, v with their windows in a pool beside the state
  pool (``conv=``; verify records per-step windows, the commit copies the accepted one);
* :data:`KDA_PAD_SLOT_ID` -- the slot id of a padding row in a batch captured in a CUDA graph per bucket.

Every call launches only on the given (or current) stream, allocates nothing beyond what the caller passes
(the wrappers allocate missing outputs and workspaces through torch), and reports device-side problems
through the workspace's status word (:func:`read_device_status`).

The binding is loaded on first use and raises if libkda has not been built.
"""
from ._binding import (  # noqa: F401
    KDA_DEVICE_BAD_COUNT, KDA_DEVICE_BAD_INDEX, KDA_DEVICE_BAD_SLOT, KDA_DEVICE_TIMEOUT, KDA_ERR_CUDA, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE,
    KDA_FINAL_TO_POOL, KDA_LOAD_INITIAL, KDA_OK, KDA_TWO_PASS, KDA_FUSED, KDA_OVERLAP, KDA_CONV_NONE, KDA_CONV_SILU, KDA_PAD_SLOT_ID, KdaError, OutputNorm, ShortConv, chunk_prefill, commit_accepted, load, make_workspace,
    prefill_schedule, prefill_workspace_size, read_device_status, recurrent_verify, spec_step, status_string, workspace_size)

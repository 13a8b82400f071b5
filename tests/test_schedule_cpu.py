"""The prefill planner's decisions, through kda_prefill_schedule (host only: these run without a GPU).

The schedules pinned here are the ones the GPU tests and the bench exercise: the plain schedule for 2048 x 8, the
plain schedule with the value-split state pass for 8192 x 4, the split schedule for the long sequences of
8192 x 3, 16384 x 1 and 16384 + 16 varlen, and the fused kernel for one-chunk sequences within one wave."""
import numpy as np
import pytest

import kda_linear_attention_bounded_gb300 as kda
from kda_linear_attention_bounded_gb300 import inputs

SMS = 152   # GB300


def cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def sched(lens_or_cu, H=16, **kw):
    c = lens_or_cu if kw.pop("is_cu", False) else cu(lens_or_cu)
    return kda.prefill_schedule(c, H, sms=SMS, **kw)


def test_bench_workloads():
    assert sched([2048] * 8) == {"kind": "plain", "value_split": False, "segments": 0, "split_sequences": 0}
    assert sched([8192] * 4) == {"kind": "plain", "value_split": True, "segments": 0, "split_sequences": 0}
    s = sched(inputs.varlen_16384_plus_16().cu_seqlens, is_cu=True)
    assert s["kind"] == "split" and s["split_sequences"] == 1 and not s["value_split"] and s["segments"] >= 2
    assert sched([256], H=2) == {"kind": "plain", "value_split": True, "segments": 0, "split_sequences": 0}


def test_long_sequences_take_the_split_schedule():
    s = sched([16384])
    assert s["kind"] == "split" and s["value_split"] and s["split_sequences"] == 1
    s = sched([8192] * 3)   # 48 pairs: the split stays ahead of the plain schedule
    assert s["kind"] == "split" and s["split_sequences"] == 3 and not s["value_split"]
    s = sched([12000] * 4)  # beyond 160 chunks the split stays ahead as well
    assert s["kind"] == "split" and s["split_sequences"] == 4
    assert sched([4000] * 4)["kind"] == "plain"   # fewer than 64 chunks: never split


def test_one_chunk_sequences_take_the_fused_kernel_within_one_wave():
    assert sched([64] * 9)["kind"] == "fused"            # 144 (sequence, head) pairs
    assert sched([64] * 10)["kind"] == "plain"           # 160 pairs: more than one wave
    assert sched([65] * 2)["kind"] == "plain"            # two chunks
    assert sched([64] * 2, conv=True)["kind"] == "plain"  # the fused kernel has no short convolutions
    assert sched([64] * 2, lower_bound=-6.0)["kind"] == "plain"   # nor the 16-row sub-blocks


def test_forced_paths():
    assert sched([8192] * 4, path="two_pass")["kind"] == "plain"
    assert sched([2048] * 8, path="fused")["kind"] == "fused"
    s = sched([2048] * 8, path="overlap")   # the lane: as many sequences as fit half the SMs (76 // 16 = 4)
    assert s["kind"] == "split" and s["split_sequences"] == 4
    with pytest.raises(kda.KdaError) as e:
        sched([2048] * 8, path="fused", conv=True)
    assert e.value.status == kda.KDA_ERR_UNSUPPORTED


def test_workspace_without_scratch_keeps_the_plain_schedule():
    # 6001 + 1 tokens: the blocks fill the workspace's bound exactly (95 chunks), so without the scratch states
    # the long sequence's state pass cannot be split
    lens = [6001, 1]
    full = kda.prefill_workspace_size(6002, 2, 16)
    no_scratch = full - 2 * 16 * 128 * 128 * 4
    assert sched(lens)["kind"] == "split"
    assert sched(lens, workspace_bytes=no_scratch)["kind"] == "plain"
    with pytest.raises(kda.KdaError) as e:   # forced, the split needs the scratch
        sched(lens, workspace_bytes=no_scratch, path="overlap")
    assert e.value.status == kda.KDA_ERR_WORKSPACE
    with pytest.raises(kda.KdaError) as e:   # less than the blocks
        sched(lens, workspace_bytes=no_scratch - 1)
    assert e.value.status == kda.KDA_ERR_WORKSPACE


def test_bad_arguments():
    for c, H, kw in ((np.array([1, 64], np.int32), 16, {}), (np.array([0, 64, 32], np.int32), 16, {}),
                     (cu([64]), 0, {}), (cu([64]), 16, {"lower_bound": 1.0})):
        with pytest.raises(kda.KdaError):
            kda.prefill_schedule(c, H, sms=SMS, **kw)

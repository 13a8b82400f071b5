"""Parity of kda_chunk_prefill (CUDA, through the C ABI) with the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from kda_linear_attention_bounded_gb300 import inputs
import kda_linear_attention_bounded_gb300 as kda
from gpu_helpers import DevicePrefill, check_out, check_state

pytestmark = pytest.mark.gpu


def _run_and_check(dev, inp, ref, path, heads=None):
    """One call on `path` (the pool first reset to the inputs' own), checked against the oracle's (ref_out, ref_S)."""
    if dev.pool is not None:
        dev.pool.copy_(torch.from_numpy(inp.pool).cuda())
    pool_before = dev.pool.clone() if dev.pool is not None else None
    ws = dev.workspace()
    out, final = dev.run(workspace=ws, path=path)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    ref_out, ref_S = ref
    hb, he = heads or (0, inp.H)
    tag = f"{inp.name} [{path or 'default'} path]"
    check_out(out[:, hb:he], ref_out[:, hb:he], f"{tag} outputs", segments=inp.cu_seqlens)
    if inp.final_to_pool:
        got = dev.pool[torch.from_numpy(inp.slot_ids).long().cuda()]
        check_state(got[:, hb:he], ref_S[:, hb:he], f"{tag} final states (pool)")
        untouched = np.setdiff1d(np.arange(inp.pool.shape[0]), inp.slot_ids)
        idx = torch.from_numpy(untouched).long().cuda()
        assert torch.equal(dev.pool[idx], pool_before[idx]), "pool slots not in slot_ids were modified"
        final = got.clone()
    else:
        check_state(final[:, hb:he], ref_S[:, hb:he], f"{tag} final states")
        if pool_before is not None:
            assert torch.equal(dev.pool, pool_before), "pool modified without KDA_FINAL_TO_POOL"
    return out, final


def _parity(inp, token_pad=0, heads=None, path=None):
    dev = DevicePrefill(inp, token_pad=token_pad)
    ref_out, ref_S, _ = oracle.run_prefill(inp, heads=heads)
    return _run_and_check(dev, inp, (ref_out, ref_S), path, heads)


def _parity_paths(inp, paths):
    """Every path in `paths` against one oracle run; returns {path: (out, final states)}."""
    dev = DevicePrefill(inp)
    ref_out, ref_S, _ = oracle.run_prefill(inp)
    return {p: _run_and_check(dev, inp, (ref_out, ref_S), p) for p in paths}


@pytest.mark.parametrize("path", [None, "two_pass", "fused"])
def test_tiny_1x256_h2(path):
    _parity(inputs.tiny_prefill(), path=path)


PATHS = ["two_pass", "fused", "overlap"]   # every execution path forced (the library picks one by shape)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("lens", [[1], [63], [64], [65], [1, 63, 64, 65, 130, 0, 200], [0, 0, 3]])
def test_varlen_ragged_pool_in(lens, path):
    inp = inputs.prefill_inputs("ragged", lens, 4, seed=11 + len(lens), pool_slots=16, load_initial=True)
    _parity(inp, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_varlen_final_to_pool_inplace(path):
    inp = inputs.prefill_inputs("inplace", [100, 7, 256], 3, seed=21, pool_slots=8, load_initial=True,
                                final_to_pool=True)
    _parity(inp, path=path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", ["weak_gate", "weak_bound", "bound_-10", "bound_0"])
def test_decay_regimes(case, path):
    kw = dict(weak_gate=dict(g_mean=-8.0), weak_bound=dict(lower_bound=-0.05),
              **{"bound_-10": dict(lower_bound=-10.0), "bound_0": dict(lower_bound=0.0)})[case]
    if path == "fused" and case == "bound_-10":
        pytest.skip("the fused kernel takes lower_bound >= -5")
    inp = inputs.prefill_inputs(case, [300, 77], 4, seed=31, pool_slots=4, load_initial=True, **kw)
    _parity(inp, path=path)


@pytest.mark.parametrize("lb", [-5.0, -5.1, -10.0])
def test_saturated_gate_at_the_sub_block_switch(lb):
    # gate pushed to its bound (lambda = lower_bound on every channel): at -5 the 32-row sub-blocks and at
    # -10 the 16-row ones see their largest exponents (2^+-115); at -5.1 the kernel takes the 16-row ones
    inp = inputs.prefill_inputs(f"saturated_{lb}", [200, 64, 33], 2, seed=35, pool_slots=4, load_initial=True,
                                lower_bound=lb, g_mean=8.0)
    _parity(inp)
    if lb >= -5.0:
        _parity(inp, path="fused")


@pytest.mark.parametrize("path", PATHS)
def test_strided_token_rows(path):
    inp = inputs.prefill_inputs("strided", [130, 64], 2, seed=41)
    _parity(inp, token_pad=256, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_bad_slot_sets_status_and_skips(path):
    inp = inputs.prefill_inputs("badslot", [70, 50], 2, seed=51, pool_slots=4, load_initial=True)
    dev = DevicePrefill(inp)
    dev.slots[1] = 99
    ws = dev.workspace()
    out = torch.full((inp.total_tokens, 2, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    out, final = dev.run(workspace=ws, out=out, path=path)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) & kda.KDA_DEVICE_BAD_SLOT
    ref_out, ref_S, _ = oracle.run_prefill(inp)
    check_out(out[:70], ref_out[:70], "good sequence next to a bad slot", segments=[0, 70])
    assert (out[70:].float() == 7.0).all(), "skipped sequence must not be written"


@pytest.mark.parametrize("make", [inputs.prefill_2048x8, inputs.prefill_8192x4, inputs.varlen_16384_plus_16],
                         ids=["2048x8", "8192x4", "16384+16varlen"])
def test_full_size(make):
    # every path against one oracle run: the library's own pick, the fused one-kernel path (KDA_FUSED), the
    # two-kernel path (KDA_TWO_PASS) and the two kernels with split state passes (KDA_OVERLAP; on 2048 x 8 four
    # of the eight sequences are split, the other four take the plain schedule beside them)
    res = _parity_paths(make(), [None, "fused", "two_pass", "overlap"])
    for p in ("overlap", None):
        assert torch.equal(res[p][0], res["two_pass"][0]) and torch.equal(res[p][1], res["two_pass"][1]), \
            f"{p or 'default'} path differs from the two-kernel path's bits"


@pytest.mark.parametrize("lens", [[1, 63, 64, 65, 130, 0, 200], [1000, 3, 700]])
def test_fused_and_two_pass_paths_agree(lens):
    # both paths on the same ragged batch: each within the bar of the oracle, and close to one another
    inp = inputs.prefill_inputs("paths", lens, 4, seed=17, pool_slots=12, load_initial=True)
    out_f, fin_f = _parity(inp, path="fused")
    out_t, fin_t = _parity(inp, path="two_pass")
    assert float((out_f.float() - out_t.float()).abs().max()) <= 3e-2
    assert float((fin_f - fin_t).norm() / fin_t.norm()) <= 5e-3


@pytest.mark.parametrize("decay", ["weak_bound", "weak_gate"])
@pytest.mark.parametrize("lens", [[8192] * 4, [16384]], ids=["8192x4", "16384x1"])
def test_full_length_weak_decay(lens, decay):
    # Weak decay over 128 or 256 chunks: with lower_bound -0.05, or the gate logits centred at -8 (lambda ~ -1e-3
    # per step), the state keeps what enters it for thousands of tokens, so an error the state path makes in one
    # chunk (the rounding of the state the products read, a wrong carry, a state handed between segments of a
    # split state pass) reaches the final state and every later output instead of being forgotten within a few
    # tokens as at the workloads' decay.
    kw = dict(weak_bound=dict(lower_bound=-0.05), weak_gate=dict(g_mean=-8.0))[decay]
    inp = inputs.prefill_inputs(f"{decay}_{len(lens)}x{lens[0]}", lens, 16, seed=90 + len(lens), pool_slots=16,
                                load_initial=True, final_to_pool=len(lens) > 1, **kw)
    _parity_paths(inp, PATHS)


@pytest.mark.parametrize("lens,H", [([5000, 300, 2000, 64, 1, 4500, 0], 16), ([700, 64, 129], 2), ([20000], 1)],
                         ids=["mixed_h16", "short_h2", "20000x1_h1"])
@pytest.mark.parametrize("final_to_pool", [False, True])
def test_overlap_schedule_matches_two_pass_bit_for_bit(lens, H, final_to_pool):
    # The split schedule runs the kernels of the two-kernel path; the state a segment hands to the next passes
    # through fp32 memory and is turned into the same operands the unsplit state pass keeps on chip, so every
    # output and final state must agree bit for bit.  mixed_h16: forced, four sequences are split (the budget of
    # half the SMs at H = 16) and the others run beside them on the plain schedule; by default only the two of
    # at least half the longest's 79 chunks are split.  short_h2: segments of 4 and then 1-4 chunks.
    inp = inputs.prefill_inputs("overlap_bits", lens, H, seed=19, pool_slots=12, load_initial=True,
                                final_to_pool=final_to_pool)
    dev = DevicePrefill(inp)
    pool0 = dev.pool.clone()
    res = {}
    for path in ("two_pass", "overlap", None):
        dev.pool.copy_(pool0)
        ws = dev.workspace()
        out, final = dev.run(workspace=ws, path=path)
        torch.cuda.synchronize()
        assert kda.read_device_status(ws) == 0
        res[path] = (out.clone(), (dev.pool if final_to_pool else final).clone())
    for path in ("overlap", None):
        assert torch.equal(res[path][0], res["two_pass"][0]), f"{path or 'default'}: outputs differ"
        assert torch.equal(res[path][1], res["two_pass"][1]), f"{path or 'default'}: final states differ"
    # and the two-kernel path itself against the oracle
    _parity(inp, path="two_pass")


def test_overlap_schedule_with_segments_over_several_intra_launches():
    # H = 1, 78 sequences of 9300 tokens: forced, 76 sequences are split (half the SMs) into segments of 55,
    # 55 and 36 chunks, so a segment holds 76 x 55 = 4180 chunk slots and its intra-chunk work takes two
    # launches (each a programmatic dependent of the one before, with its own counter); the other two
    # sequences' chunks join those launches.  Bit for bit against the two-kernel path.
    inp = inputs.prefill_inputs("overlap_runs", [9300] * 78, 1, seed=29, pool_slots=80, load_initial=True)
    dev = DevicePrefill(inp)
    res = {}
    for path in ("two_pass", "overlap"):
        ws = dev.workspace()
        out, final = dev.run(workspace=ws, path=path)
        torch.cuda.synchronize()
        assert kda.read_device_status(ws) == 0
        res[path] = (out.clone(), final.clone())
    assert torch.equal(res["overlap"][0], res["two_pass"][0])
    assert torch.equal(res["overlap"][1], res["two_pass"][1])


def test_overlap_workspace_without_scratch_takes_the_plain_schedule():
    # a workspace with the blocks but not the scratch states (for these lengths the blocks' bound is exact, so no
    # spare block holds a scratch state): the call runs unsplit and gives the same bits
    inp = inputs.prefill_inputs("overlap_ws", [6001, 1], 4, seed=23)
    dev = DevicePrefill(inp)
    full = kda.prefill_workspace_size(inp.total_tokens, inp.num_seqs, inp.H)
    scratch = min(inp.num_seqs * inp.H, 96) * 128 * 128 * 4
    ref, _ = dev.run(workspace=dev.workspace(), path="two_pass")
    small = kda.make_workspace("cuda", nbytes=full - scratch)
    out, _ = dev.run(workspace=small)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    with pytest.raises(kda.KdaError):   # forced, the split needs the scratch
        dev.run(workspace=small, path="overlap")


@pytest.mark.parametrize("path", [None] + PATHS)
@pytest.mark.parametrize("H", [3, 5, 32])
def test_head_counts_outside_the_bench_shapes(H, path):
    # odd head counts (a grid of chunk slots x H CTAs, value-split pairs of CTAs over (sequence, head)) and a
    # larger one; ragged lengths with an empty and a one-token sequence, pool in and out
    inp = inputs.prefill_inputs(f"heads_{H}", [200, 65, 0, 1, 130], H, seed=80 + H, pool_slots=7,
                                load_initial=True, final_to_pool=True)
    _parity(inp, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_more_sequences_than_one_launch_plans(path):
    # 1100 sequences: the planner splits them into two launch groups of <= 1024 sequences
    rng = np.random.default_rng(61)
    lens = [int(x) for x in rng.integers(0, 40, size=1100)]
    inp = inputs.prefill_inputs("many_seqs", lens, 2, seed=62, pool_slots=1100, load_initial=True,
                                final_to_pool=True)
    _parity(inp, path=path)


def test_more_chunk_slots_than_one_intra_launch():
    # 80 sequences of 3000..4000 tokens, H = 1: about 4400 chunk slots, so the intra-chunk work is split over
    # two launches and the second one starts inside a sequence
    rng = np.random.default_rng(71)
    lens = [int(x) for x in rng.integers(3000, 4001, size=80)]
    inp = inputs.prefill_inputs("many_slots", lens, 1, seed=72, pool_slots=96, load_initial=True)
    assert sum((n + 63) // 64 for n in lens) > 4096
    _parity(inp)


@pytest.mark.parametrize("path", PATHS)
def test_prefill_captured_in_a_cuda_graph(path):
    # the call (intra-chunk launch + state pass as its programmatic dependent) replays from a CUDA graph with
    # the same results as a direct call
    inp = inputs.prefill_inputs("graph", [130, 64, 200, 1], 2, seed=81, pool_slots=8, load_initial=True)
    dev = DevicePrefill(inp)
    ws = dev.workspace()
    out_ref, final_ref = dev.run(workspace=ws, path=path)
    torch.cuda.synchronize()
    out_ref, final_ref = out_ref.clone(), final_ref.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        dev.run(workspace=ws, path=path)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out_g, final_g = dev.run(workspace=ws, path=path)
    out_g.zero_()
    final_g.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    assert torch.equal(out_g, out_ref)
    assert torch.equal(final_g, final_ref)


def test_concurrent_calls_from_two_threads():
    # two host threads, each with its own stream and workspace, call the prefill at once (the planner's staging
    # of the launch parameters is shared and locked; the split schedule's counters live in each workspace): both
    # give the results of a call made alone, bit for bit
    import threading
    inps = [inputs.prefill_inputs("thread_a", [5000, 300], 4, seed=33, pool_slots=4, load_initial=True),
            inputs.prefill_inputs("thread_b", [700, 64, 129], 4, seed=34, pool_slots=4, load_initial=True)]
    devs = [DevicePrefill(i) for i in inps]
    refs = []
    for d in devs:
        out, fin = d.run(workspace=d.workspace())
        torch.cuda.synchronize()
        refs.append((out.clone(), fin.clone()))
    results = [None, None]
    errors = []

    def work(k):
        try:
            st = torch.cuda.Stream()
            ws = devs[k].workspace()
            torch.cuda.synchronize()
            with torch.cuda.stream(st):
                for _ in range(5):
                    out, fin = devs[k].run(workspace=ws, stream=st)
            st.synchronize()
            assert kda.read_device_status(ws, stream=st) == 0
            results[k] = (out.clone(), fin.clone())
        except Exception as e:   # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for k in range(2):
        assert torch.equal(results[k][0], refs[k][0]) and torch.equal(results[k][1], refs[k][1])


@pytest.mark.parametrize("seed", range(8))
def test_schedules_agree_bit_for_bit_on_random_shapes(seed):
    # Seeded random workloads: 1..12 sequences of 0..6000 tokens (empty, one-token and non-multiples of 64
    # included), H in {1, 2, 4, 16}, lower_bound in [-10, -0.05], pool or zero initial states, dense or
    # in-place final states, every third one with the short convolutions.  The library's own pick (which takes
    # the split schedule and the value-split state pass where they apply) and the forced split schedule must
    # give the two-kernel path's bits; the two-kernel path itself is held to the oracle on two heads.
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(1, 13))
    lens = [int(x) for x in rng.integers(0, 6001, size=n)]
    for i in range(n):
        r = rng.random()
        lens[i] = 0 if r < 0.08 else 1 if r < 0.14 else lens[i]
    if sum(lens) == 0:
        lens[0] = 65
    H = int(rng.choice([1, 2, 4, 16]))
    lb = float(-10 ** rng.uniform(np.log10(0.05), 1.0))
    load_initial = bool(rng.random() < 0.6)
    final_to_pool = load_initial and bool(rng.random() < 0.5)
    inp = inputs.prefill_inputs(f"random_{seed}", lens, H, seed=2000 + seed, pool_slots=n + 2,
                                load_initial=load_initial, final_to_pool=final_to_pool, lower_bound=lb)
    conv = None
    if seed % 3 == 2:
        from gpu_helpers import device_conv
        inp.conv = inputs.conv_inputs(H, n + 2, seed=3000 + seed)
    dev = DevicePrefill(inp)
    pool0 = dev.pool.clone() if dev.pool is not None else None
    res = {}
    for path in ("two_pass", None, "overlap"):
        if pool0 is not None:
            dev.pool.copy_(pool0)
        kw = {}
        if inp.conv is not None:
            conv = device_conv(inp.conv, N=None if final_to_pool else inp.num_seqs)
            kw["conv"] = conv
        ws = dev.workspace()
        out, final = dev.run(workspace=ws, path=path, **kw)
        torch.cuda.synchronize()
        assert kda.read_device_status(ws) == 0
        win = None if conv is None else (conv.window_pool if final_to_pool else conv.window_dense).clone()
        res[path] = (out.clone(), (dev.pool if final_to_pool else final).clone(), win)
    for path in (None, "overlap"):
        for a, b, what in zip(res[path], res["two_pass"], ("outputs", "final states", "windows")):
            if a is not None:
                assert torch.equal(a, b), f"{path or 'default'} path: {what} differ from the two-kernel path's"
    if inp.conv is None:
        hb = min(2, H)
        ref_out, ref_S, _ = oracle.run_prefill(inp, heads=(0, hb))
        check_out(res["two_pass"][0][:, :hb], ref_out[:, :hb], f"{inp.name} outputs", segments=inp.cu_seqlens)
        got = res["two_pass"][1]
        if final_to_pool:
            got = got[torch.from_numpy(inp.slot_ids).long().cuda()]
        check_state(got[:, :hb], ref_S[:, :hb], f"{inp.name} final states")

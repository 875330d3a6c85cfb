"""fused_qk_norm_rope on the GPU against the oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import kv_quant_cache_gb300 as kvq
import workloads as wl
from gpu_cases import qk_parity, qk_parity_sampled, to_device, with_config

pytestmark = pytest.mark.gpu


def test_decode_size_17_tokens(cuda_device, parity_log):
    rep = qk_parity(wl.make_qk_workload(wl.QK_SMALL, device=cuda_device))
    assert rep.exact_frac > 0.95
    parity_log(rep)


@pytest.mark.parametrize("config", [-1, 7, 10], ids=["auto", "bulk", "tile"])
def test_prefill_32768_tokens_every_token(cuda_device, config, parity_log):
    """The benchmarked workload, compared in full (1,310,720 head rows), under
    the automatic dispatch and under a TMA-staged shape."""
    with with_config("qk", config):
        rep = qk_parity(wl.make_qk_workload(wl.QK_LARGE, device=cuda_device), slice_tokens=8192)
    assert rep.n == 32768 * 40 * 128
    assert rep.exact_frac > 0.95
    parity_log(rep)


@pytest.mark.parametrize("T", [1, 4, 17, 511, 512, 777, 1000, 4096])
@pytest.mark.parametrize("heads", [(16, 8, 8), (3, 2, 1), (5, 0, 2), (0, 3, 0), (1, 1, 0),
                                   (32, 8, 8)])
def test_ragged_shapes(cuda_device, T, heads):
    """Token counts that are not multiples of any tile, odd Q+K counts, no K,
    no Q, no V: both launch shapes (the small one below 1216 rows)."""
    Hq, Hk, Hv = heads
    d = wl.make_qk(T, Hq, Hk, Hv, theta=1e6, max_pos=131072, seed=T * 7 + Hq,
                   device=cuda_device)
    qk_parity(d)


def test_positions_at_table_edges(cuda_device):
    d = wl.make_qk(64, 4, 2, 2, theta=1e4, max_pos=4096, seed=5, device=cuda_device)
    d["positions"] = torch.tensor([0, 4095] * 32, dtype=torch.int64, device=cuda_device)
    qk_parity(d)


def test_exact_arithmetic_rows(cuda_device):
    """x = +-1 everywhere, eps = 0 and position 0: r = 1 exactly and the
    rotation is the identity, so every output is w rounded to bf16 -- bit-exact."""
    T, Hq, Hk, Hv = 9, 2, 2, 1
    rng = np.random.default_rng(1)
    sign = np.where(rng.random((T, (Hq + Hk + Hv) * 128)) < 0.5, -1.0, 1.0)
    d = wl.make_qk(T, Hq, Hk, Hv, max_pos=8, seed=2, device="cpu", eps=0.0)
    d["qkv"] = wl.bf16_from_values(sign)
    d["positions"] = torch.zeros(T, dtype=torch.int64)
    rep = qk_parity(to_device(d, cuda_device))
    assert rep.exact == rep.n


def test_zero_rows_and_tiny_values(cuda_device):
    """All-zero heads (r = 1/sqrt(eps)) and values far below 1 stay finite and match."""
    d = wl.make_qk(16, 4, 4, 0, max_pos=64, seed=3, device="cpu")
    x = d["qkv"].float()
    x[0:4] = 0.0
    x[4:8] *= 1e-30
    x[8:12] *= 1e6
    d["qkv"] = x.to(torch.bfloat16)
    qk_parity(to_device(d, cuda_device))


@pytest.mark.parametrize("config", [-1, 2, 5, 7], ids=["auto", "tiles4", "general", "bulk"])
def test_eps_zero_all_zero_rows_are_nan(cuda_device, config):
    """eps = 0: an all-zero head row has no norm (0/0).  The oracle gives NaN
    there and so must every launch family; the other rows match the oracle
    and V is untouched."""
    import oracle
    from parity import Bf16Report
    T, Hq, Hk, Hv, D = 24, 4, 2, 2, 128
    d = wl.make_qk(T, Hq, Hk, Hv, max_pos=64, seed=21, device="cpu", eps=0.0)
    x = d["qkv"].float()
    x[[3, 17]] = 0.0
    d["qkv"] = x.to(torch.bfloat16)
    inp = wl.bf16_bits(d["qkv"])
    g = to_device(d, cuda_device)
    with with_config("qk", config):
        kvq.fused_qk_norm_rope(g["qkv"], Hq, Hk, Hv, D, 0.0, g["q_weight"], g["k_weight"],
                               g["cos_sin"], True, g["positions"])
    torch.cuda.synchronize()
    gpu = wl.bf16_bits(g["qkv"]).reshape(T, Hq + Hk + Hv, D)
    out, ref, mag = oracle.qk_norm_rope(inp, Hq, Hk, Hv, D, 0.0, wl.bf16_bits(d["q_weight"]),
                                        wl.bf16_bits(d["k_weight"]), wl.host(d["cos_sin"]),
                                        wl.host(d["positions"]), want_ref=True)
    out = out.reshape(T, Hq + Hk + Hv, D)
    NR = Hq + Hk

    def isnan(b):
        return ((b & 0x7f80) == 0x7f80) & ((b & 0x7f) != 0)
    zero = np.zeros(T, bool)
    zero[[3, 17]] = True
    assert isnan(out[zero, :NR]).all() and isnan(gpu[zero, :NR]).all()
    assert not isnan(gpu[~zero, :NR]).any()
    assert np.array_equal(gpu[:, NR:], inp.reshape(T, -1, D)[:, NR:])
    rep = Bf16Report()
    rep.add(gpu[~zero, :NR], out[~zero, :NR], ref[~zero], mag[~zero])
    rep.check("fused_qk_norm_rope, eps = 0")


def test_zero_tokens_is_a_no_op(cuda_device):
    d = wl.make_qk(0, 2, 1, 1, device=cuda_device)
    kvq.fused_qk_norm_rope(d["qkv"], 2, 1, 1, 128, 1e-6, d["q_weight"], d["k_weight"],
                           d["cos_sin"], True, d["positions"])
    torch.cuda.synchronize()


def test_runs_on_a_side_stream(cuda_device):
    d = wl.make_qk(300, 8, 4, 4, max_pos=4096, seed=9, device=cuda_device)
    s = torch.cuda.Stream(cuda_device)
    ref = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        kvq.fused_qk_norm_rope(d["qkv"], 8, 4, 4, 128, 1e-6, d["q_weight"], d["k_weight"],
                               d["cos_sin"], True, d["positions"], stream=s)
    s.synchronize()
    qk_parity(ref)  # the same inputs through the default stream
    assert torch.equal(d["qkv"], ref["qkv"])


QK_CONFIGS = list(range(11))


@pytest.mark.parametrize("config", QK_CONFIGS)
@pytest.mark.parametrize("shape", [(1, 16, 8, 8), (777, 5, 3, 2), (300, 32, 8, 8), (64, 1, 0, 1)])
def test_every_launch_config(cuda_device, config, shape):
    """Each launch shape of the table against the oracle (forced), on ragged
    token counts and head counts that leave partial chunks."""
    assert len(kvq.configs("qk")) == len(QK_CONFIGS)
    T, Hq, Hk, Hv = shape
    d = wl.make_qk(T, Hq, Hk, Hv, theta=1e6, max_pos=131072, seed=31 + config, device=cuda_device)
    with with_config("qk", config):
        qk_parity(d)


LAYOUTS = [(D, rot, neox) for D in (64, 128, 256) for neox in (True, False)
           for rot in sorted({16, D // 2, D}) if rot % 16 == 0 and not (D == 128 and rot == 128 and neox)]


@pytest.mark.parametrize("config", [-1, 5, 6, 7, 8, 9, 10],
                         ids=["auto", "frag4", "frag8", "bulk6KB", "bulk3KB", "bulk2KB", "tile6KB"])
@pytest.mark.parametrize("layout", LAYOUTS, ids=lambda l: f"D{l[0]}_rot{l[1]}_{'neox' if l[2] else 'gptj'}")
@pytest.mark.parametrize("shape", [(1, 4, 2, 1), (17, 3, 1, 2), (777, 8, 2, 2), (300, 0, 5, 0)])
def test_general_layouts(cuda_device, layout, shape, config):
    """head_dim 64/128/256, NeoX or GPT-J pairs, full or partial rotation,
    through the one-shot general kernel (automatic choice, 4- and 8-dim
    fragments forced) and the TMA-staged shapes, against the oracle."""
    assert kvq.configs("qk")[5:7] == ["general<frag4>", "general<frag8>"]
    D, rot, neox = layout
    T, Hq, Hk, Hv = shape
    d = wl.make_qk(T, Hq, Hk, Hv, D=D, theta=1e4, max_pos=8192, seed=D + rot + T,
                   device=cuda_device, rotary_dim=rot, is_neox=neox)
    with with_config("qk", config):
        qk_parity(d)


def test_general_layout_at_scale(cuda_device):
    """A 32768-token partial-rotation GPT-J case (the general kernel's large
    launch), every token against the oracle."""
    d = wl.make_qk(32768, 16, 4, 4, D=256, theta=1e6, max_pos=131072, seed=77,
                   device=cuda_device, rotary_dim=64, is_neox=False)
    qk_parity(d, slice_tokens=8192)


BULK = list(range(7, 11))   # the TMA-staged shapes (the last one tiled)
# The 4-dim-fragment shapes of the D=128 NeoX layout, in their two groups:
# the register-pipelined and one-shot shapes (hardware reciprocal square
# root) and the TMA-staged shapes (correctly rounded one).
ONE_SHOT_SHAPES = [0, 1, 2, 3, 4, 5]


def _groups_agree(a, b, what=""):
    """Results of the two shape groups: equal bits except for rare values (an
    fp32 value next to a bf16 rounding boundary, or a rotation that cancels);
    each group is also checked against the oracle."""
    frac = float((a != b).float().mean().item())
    assert frac < 1e-4, (what, frac)


def _run_config(d, config):
    out = d["qkv"].clone()
    with with_config("qk", config):
        kvq.fused_qk_norm_rope(out, d["Hq"], d["Hk"], d["Hv"], 128, d["eps"], d["q_weight"],
                               d["k_weight"], d["cos_sin"], True, d["positions"])
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("shape", [(4096, 32, 8, 8), (777, 5, 3, 2), (1, 16, 8, 8),
                                   (300, 64, 8, 8), (50, 100, 28, 3)])
def test_launch_shapes_bit_identical(cuda_device, shape):
    """The register-pipelined and one-shot general shapes share the row
    arithmetic and the lane mapping: every one gives the same bits; so do the
    TMA-staged shapes among themselves.  Between the two groups (approximate
    vs correctly rounded reciprocal square root) at most rare values differ,
    by one bf16 ulp."""
    assert [n.startswith("bulk") for n in kvq.configs("qk")] == [False] * 7 + [True] * 4
    T, Hq, Hk, Hv = shape
    d = wl.make_qk(T, Hq, Hk, Hv, theta=1e6, max_pos=131072, seed=T + Hq, device=cuda_device)
    ref = _run_config(d, 2)
    assert not torch.equal(ref, d["qkv"])
    for config in ONE_SHOT_SHAPES:
        assert torch.equal(_run_config(d, config), ref), kvq.configs("qk")[config]
    staged = _run_config(d, BULK[0])
    for config in BULK:
        assert torch.equal(_run_config(d, config), staged), kvq.configs("qk")[config]
    _groups_agree(staged, ref, "staged vs one-shot")
    for config in (2, BULK[0]):
        with with_config("qk", config):
            qk_parity({k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in d.items()})


@pytest.mark.parametrize("config", BULK)
def test_staged_shape_finishing_from_global_memory(cuda_device, config):
    """With a stage-wait limit of 0 every warp of a staged launch gives up on
    its first wait: it lets its copies land, then finishes every item with
    direct loads.  The results are the same bits, and match the oracle."""
    d = wl.make_qk(2000, 32, 8, 8, theta=1e6, max_pos=131072, seed=61, device=cuda_device)
    ref = _run_config(d, BULK[0])
    kvq.stage_events(reset=True)
    assert _run_config(d, config).equal(ref)     # default limit: nothing falls back
    assert kvq.stage_events(reset=True) == (0, 0)
    old = kvq.set_stage_wait_limit(0)
    try:
        assert old > 0
        assert torch.equal(_run_config(d, config), ref)
        fallbacks, drain_timeouts = kvq.stage_events(reset=True)
        # every warp with items reports its fallback; each drained its copies
        assert fallbacks >= 1 and drain_timeouts == 0, (fallbacks, drain_timeouts)
        with with_config("qk", config):
            qk_parity(d)
    finally:
        kvq.set_stage_wait_limit(old)
    assert kvq.set_stage_wait_limit(old) == old
    assert kvq.stage_events(reset=True)[1] == 0


def _run_layout(d, config):
    out = d["qkv"].clone()
    with with_config("qk", config):
        kvq.fused_qk_norm_rope(out, d["Hq"], d["Hk"], d["Hv"], d["D"], d["eps"], d["q_weight"],
                               d["k_weight"], d["cos_sin"], d["is_neox"], d["positions"],
                               rotary_dim=d["rot"])
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("layout", [l for l in LAYOUTS if l[1] < l[0] or not l[2]],
                         ids=lambda l: f"D{l[0]}_rot{l[1]}_{'neox' if l[2] else 'gptj'}")
def test_general_staged_bit_identical(cuda_device, layout):
    """Every TMA-staged shape gives the same bits for every layout (shared row
    arithmetic and lane mapping); the one-shot general kernel, on the
    approximate reciprocal square root, agrees with them up to rare values
    one bf16 ulp apart."""
    D, rot, neox = layout
    d = wl.make_qk(1500, 24, 8, 4, D=D, theta=1e6, max_pos=131072, seed=D * 3 + rot,
                   device=cuda_device, rotary_dim=rot, is_neox=neox)
    ref = _run_layout(d, BULK[0])
    for config in BULK:
        assert torch.equal(_run_layout(d, config), ref), kvq.configs("qk")[config]
    _groups_agree(_run_layout(d, 5), ref, "general vs staged")


@pytest.mark.parametrize("layout", [(64, 32, False), (256, 256, True), (256, 64, False)],
                         ids=lambda l: f"D{l[0]}_rot{l[1]}_{'neox' if l[2] else 'gptj'}")
def test_general_staged_finishing_from_global_memory(cuda_device, layout):
    """Stage-wait limit 0 on the general layouts: every warp drains its copies
    and finishes from global memory, with the same bits."""
    D, rot, neox = layout
    d = wl.make_qk(900, 16, 4, 4, D=D, theta=1e6, max_pos=131072, seed=D + rot + 1,
                   device=cuda_device, rotary_dim=rot, is_neox=neox)
    ref = _run_layout(d, BULK[0])
    kvq.stage_events(reset=True)
    old = kvq.set_stage_wait_limit(0)
    try:
        for config in BULK:
            assert torch.equal(_run_layout(d, config), ref), kvq.configs("qk")[config]
            fallbacks, drain_timeouts = kvq.stage_events(reset=True)
            assert fallbacks >= 1 and drain_timeouts == 0, (config, fallbacks, drain_timeouts)
    finally:
        kvq.set_stage_wait_limit(old)


def test_staged_shape_at_131072_tokens(cuda_device):
    """The largest QK workload of the sweep (131072 tokens, 5.2M head rows:
    the staged shape's regime), every token against the oracle; no warp
    stopped staging."""
    d = wl.make_qk(131072, 32, 8, 8, theta=1e6, max_pos=131072, seed=1001, device=cuda_device)
    assert kvq.configs("qk")[kvq.qk_config_for(131072, 32, 8)].startswith("bulk")
    kvq.stage_events(reset=True)
    rep = qk_parity(d, slice_tokens=16384)
    assert rep.n == 131072 * 40 * 128
    assert kvq.stage_events(reset=True) == (0, 0)


@pytest.mark.parametrize("config", [-1, 2, 4, 5, 10],
                         ids=["auto", "tiles4", "stream", "general", "tile"])
def test_offsets_beyond_4_gib(cuda_device, config, parity_log):
    """360000 tokens x 48 heads x 128 dims: qkv is 4.42 GB, so element offsets
    pass 2^31 and byte offsets 2^32.  Every launch family; the first and last
    tokens and 1024 random ones against the oracle, V unchanged everywhere."""
    T = 360000
    assert T * 48 * 128 > 2**31 and T * 48 * 128 * 2 > 2**32
    d = wl.make_qk(T, 32, 8, 8, theta=1e6, max_pos=131072, seed=4242, device=cuda_device)
    with with_config("qk", config):
        rep = qk_parity_sampled(d, 1024, seed=config + 1)
    parity_log(rep)
    del d
    torch.cuda.empty_cache()


def test_general_layout_offsets_beyond_4_gib(cuda_device, parity_log):
    """head_dim 256, GPT-J pairs, 64 rotated dims, 180000 tokens (4.42 GB of
    qkv), through the automatic (staged) shape and the one-shot kernel."""
    T = 180000
    for config in (-1, 5):
        d = wl.make_qk(T, 32, 8, 8, D=256, theta=1e6, max_pos=131072, seed=4343,
                       device=cuda_device, rotary_dim=64, is_neox=False)
        with with_config("qk", config):
            rep = qk_parity_sampled(d, 1024, seed=config + 7)
        parity_log(rep)
        del d
        torch.cuda.empty_cache()


@pytest.mark.skipif(not torch.cuda.is_available() or torch.cuda.device_count() < 2,
                    reason="needs two GPUs")
def test_tensors_on_a_device_other_than_the_current_one():
    """With the current device set to GPU 0, a call on GPU 1's tensors runs
    on GPU 1 (the binding switches for the call) and matches the oracle; a
    call mixing the two devices is refused before anything is launched."""
    dev1 = torch.device("cuda:1")
    with torch.cuda.device(0):
        d = wl.make_qk(4096, 32, 8, 8, theta=1e6, max_pos=131072, seed=91, device=dev1)
        for config in (-1, 7):
            with with_config("qk", config):
                qk_parity({k: (v.clone() if isinstance(v, torch.Tensor) else v)
                           for k, v in d.items()})
        assert torch.cuda.current_device() == 0
        with pytest.raises(ValueError):
            kvq.fused_qk_norm_rope(d["qkv"], 32, 8, 8, 128, d["eps"], d["q_weight"].to("cuda:0"),
                                   d["k_weight"], d["cos_sin"], True, d["positions"])


def test_two_streams_at_once(cuda_device):
    """Both operators enqueued on two streams at the same time (independent
    buffers, programmatic launch on) give the bytes of a run on their own;
    the QK result is also checked against the oracle."""
    from gpu_cases import dsv4_parity, run_dsv4
    qk = wl.make_qk(32768, 32, 8, 8, theta=1e6, max_pos=131072, seed=81, device=cuda_device)
    ds = wl.make_dsv4(4096, 64, max_pos=131072, num_blocks=128, block_size=64, seed=82,
                      device=cuda_device)
    ref_qk = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in qk.items()}
    ref_ds = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in ds.items()}
    s1, s2 = torch.cuda.Stream(cuda_device), torch.cuda.Stream(cuda_device)
    torch.cuda.synchronize()
    for _ in range(3):  # same inputs each time: restore, then run both at once
        qk["qkv"].copy_(ref_qk["qkv"])
        ds["q"].copy_(ref_ds["q"])
        torch.cuda.synchronize()
        with torch.cuda.stream(s1):
            kvq.fused_qk_norm_rope(qk["qkv"], 32, 8, 8, 128, qk["eps"], qk["q_weight"],
                                   qk["k_weight"], qk["cos_sin"], True, qk["positions"], stream=s1)
        with torch.cuda.stream(s2):
            kvq.dsv4_qnorm_rope_kv_rope_quant_insert(
                ds["q"], ds["kv"], ds["eps"], ds["q_weight"], ds["kv_weight"], ds["cos_sin"],
                ds["positions"], ds["slot_mapping"], ds["kv_cache"], stream=s2)
        torch.cuda.synchronize()
    got_qk, got_q, got_cache = qk["qkv"].clone(), ds["q"].clone(), ds["kv_cache"].clone()
    qk_parity(ref_qk)            # reference: one operator at a time on the default stream
    run_dsv4(ref_ds)
    torch.cuda.synchronize()
    assert torch.equal(got_qk, ref_qk["qkv"])
    assert torch.equal(got_q, ref_ds["q"]) and torch.equal(got_cache, ref_ds["kv_cache"])


def test_default_stream_is_torchs_current_stream(cuda_device):
    """Calls without `stream` enqueue on torch's current stream, also inside a
    `torch.cuda.stream` context (the binding reads the raw handle)."""
    s = torch.cuda.Stream(cuda_device)
    idx = cuda_device.index or 0
    assert kvq._stream(None, idx) == torch.cuda.current_stream(cuda_device).cuda_stream
    with torch.cuda.stream(s):
        assert kvq._stream(None, idx) == s.cuda_stream
        assert kvq._stream(None, idx) == torch.cuda.current_stream(cuda_device).cuda_stream

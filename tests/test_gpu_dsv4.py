"""dsv4_qnorm_rope_kv_rope_quant_insert on the GPU against the oracle."""
import numpy as np
import pytest
import torch

import kv_quant_cache_gb300 as kvq
import workloads as wl
from gpu_cases import (SMALL_PATH, TILED_PATH, dsv4_parity, run_dsv4, to_device, with_config,
                       with_threshold)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("threshold", [None, SMALL_PATH, TILED_PATH], ids=["auto", "small", "tiled"])
def test_decode_size_16_tokens(cuda_device, threshold, parity_log):
    """The 16-token decode workload (64 heads, two tokens without a slot)."""
    d = wl.make_dsv4_workload(wl.DSV4_DECODE, device=cuda_device)
    assert int((d["slot_mapping"] < 0).sum()) == 2
    if threshold is None:
        qrep, crep = dsv4_parity(d)
    else:
        with with_threshold(threshold):
            qrep, crep = dsv4_parity(d)
    assert crep.entries == 14
    assert crep.exp_mismatch_ties == 0
    parity_log(qrep, crep)


def test_prefill_32768x64_every_token(cuda_device, parity_log):
    """The benchmarked workload (default dispatch = the persistent launch),
    every token and the whole cache compared."""
    d = wl.make_dsv4_workload(wl.DSV4_LARGE, device=cuda_device)
    assert kvq.dsv4_dispatch_path(32768, 64) == 1
    qrep, crep = dsv4_parity(d, slice_tokens=1024)
    assert qrep.n == 32768 * 64 * 512
    assert crep.entries == 32768
    assert crep.exp_mismatch_ties == 0
    parity_log(qrep, crep)


@pytest.mark.parametrize("w", [w for w in wl.DSV4_SWEEP if w.T <= 8192], ids=lambda w: w.name)
def test_sweep_every_token(cuda_device, w, parity_log):
    qrep, crep = dsv4_parity(wl.make_dsv4_workload(w, device=cuda_device), slice_tokens=512)
    assert crep.exp_mismatch_ties == 0
    parity_log(qrep, crep)


@pytest.mark.parametrize("w", [w for w in wl.DSV4_SWEEP if w.T > 8192], ids=lambda w: w.name)
def test_sweep_full_size_sampled(cuda_device, w, parity_log):
    """Full-size launch; 1024 sampled tokens (plus the first and last 8) compared
    with the oracle, and the whole cache checked for untouched slots."""
    qrep, crep = dsv4_parity(wl.make_dsv4_workload(w, device=cuda_device), sample=1024,
                             seed=w.seed)
    assert crep.exp_mismatch_ties == 0
    parity_log(qrep, crep)


@pytest.mark.parametrize("T", [1, 4, 17, 511, 512, 777, 1000])
@pytest.mark.parametrize("threshold", [SMALL_PATH, TILED_PATH], ids=["small", "tiled"])
@pytest.mark.parametrize("H", [1, 3, 64])
def test_ragged_both_launches(cuda_device, T, threshold, H):
    """Token counts off every tile and odd head counts, forced through each launch."""
    d = wl.make_dsv4(T, H, max_pos=131072, num_blocks=-(-2 * T // 16), block_size=16,
                     slots="distinct_skip2", seed=100 + T + H, device=cuda_device)
    with with_threshold(threshold):
        dsv4_parity(d)


def test_all_tokens_unmapped(cuda_device):
    d = wl.make_dsv4(37, 2, max_pos=1024, num_blocks=4, block_size=16, seed=7, device=cuda_device)
    d["slot_mapping"].fill_(-1)
    qrep, crep = dsv4_parity(d)
    assert crep.entries == 0


@pytest.mark.parametrize("threshold", [SMALL_PATH, TILED_PATH], ids=["small", "tiled"])
def test_eps_zero_all_zero_q_rows_are_nan(cuda_device, threshold):
    """eps = 0: all-zero q rows (tokens 2 and 9, which have no cache slot)
    come out NaN, as in the oracle; every other q row and every written
    cache entry matches the oracle, and no other cache byte changes."""
    import oracle
    from parity import Bf16Report, compare_cache
    T, H = 12, 3
    d = wl.make_dsv4(T, H, max_pos=4096, num_blocks=1, block_size=32, seed=31, device="cpu",
                     eps=0.0)
    q = d["q"].float()
    q[[2, 9]] = 0.0
    d["q"] = q.to(torch.bfloat16)
    d["slot_mapping"][[2, 9]] = -1
    q_in, cache_in = wl.bf16_bits(d["q"]), wl.host(d["kv_cache"]).copy()
    g = to_device(d, cuda_device)
    with with_threshold(threshold):
        run_dsv4(g)
    torch.cuda.synchronize()
    res = oracle.dsv4(q_in, wl.bf16_bits(d["kv"]), 0.0, wl.bf16_bits(d["q_weight"]),
                      wl.bf16_bits(d["kv_weight"]), wl.host(d["cos_sin"]),
                      wl.host(d["positions"]), wl.host(d["slot_mapping"]), cache_in,
                      want_ref=True)
    gq = wl.bf16_bits(g["q"])

    def isnan(b):
        return ((b & 0x7f80) == 0x7f80) & ((b & 0x7f) != 0)
    zero = np.zeros(T, bool)
    zero[[2, 9]] = True
    assert isnan(res["q"][zero]).all() and isnan(gq[zero]).all()
    assert not isnan(gq[~zero]).any()
    rep = Bf16Report()
    rep.add(gq[~zero], res["q"][~zero], res["q_ref"][~zero], res["q_mag"][~zero])
    rep.check("dsv4 q, eps = 0")
    crep = compare_cache(wl.host(g["kv_cache"]), cache_in, wl.host(d["slot_mapping"]),
                         res["kv_ref"], res["kv_mag"], res["exp_margin"])
    crep.check("dsv4 cache, eps = 0")


def test_last_slot_and_last_position(cuda_device):
    d = wl.make_dsv4(4, 2, max_pos=4096, num_blocks=3, block_size=8, seed=8, device=cuda_device)
    d["slot_mapping"] = torch.tensor([23, 0, -1, 22], dtype=torch.int64, device=cuda_device)
    d["positions"] = torch.tensor([4095, 0, 4095, 1], dtype=torch.int64, device=cuda_device)
    dsv4_parity(d)


def _exact_case(block_w, T=3):
    """kv = q = +-1, eps = 0, position 0: r = 1 exactly and the rotation is the
    identity, so n = +-w exactly in fp32 and fp64, and every exponent and code
    decision is exact on both sides."""
    rng = np.random.default_rng(3)
    d = wl.make_dsv4(T, 2, max_pos=4, num_blocks=2, block_size=8, seed=4, device="cpu", eps=0.0)
    d["q"] = wl.bf16_from_values(np.where(rng.random((T, 2, 512)) < 0.5, -1.0, 1.0))
    d["kv"] = wl.bf16_from_values(np.where(rng.random((T, 512)) < 0.5, -1.0, 1.0))
    d["kv_weight"] = wl.bf16_from_values(block_w)
    d["positions"] = torch.zeros(T, dtype=torch.int64)
    return d


def test_exponent_boundaries_and_code_ties_exact(cuda_device):
    # block 0: amax exactly 448 * 2^-7 = 3.5 (e = -7, not -6); block 1: one bf16
    # step above 3.5 (e = -6); block 2: e4m3 midpoints after scaling (ties to
    # even); block 3: values whose scaled codes are subnormal e4m3; block 4:
    # a block of zeros (byte 0); blocks 5, 6: mixed powers of two; rotary dims.
    w = np.ones(512)
    w[0:64] = 3.5
    w[1:64:2] = -1.25
    w[64:128] = 3.515625
    w[128:192] = [1.0 + 1.0 / 16 * (k % 8) for k in range(64)]  # 17/16.. -> ties at 2^-e scale
    w[128] = 2.0 ** 3
    w[192:256] = [(k % 8 + 0.5) * 2.0 ** -17 for k in range(64)]  # subnormal e4m3 ties
    w[192] = 1.0
    w[256:320] = 0.0
    w[320:384] = [2.0 ** (k % 9 - 4) for k in range(64)]
    w[384:448] = [-(2.0 ** (-(k % 11))) for k in range(64)]
    w[448:512] = np.linspace(-2, 2, 64)
    d = to_device(_exact_case(w), cuda_device)
    qrep, crep = dsv4_parity(d)
    assert qrep.exact == qrep.n
    assert crep.codes_exact == crep.codes and crep.exp_mismatch_ties == 0
    assert crep.rope.exact == crep.rope.n
    ent = d["kv_cache"].view(-1, 584)[d["slot_mapping"][0]].cpu().numpy()
    assert ent[576] == 120 and ent[577] == 121 and ent[580] == 0


def test_zero_kv_vector(cuda_device):
    d = wl.make_dsv4(5, 2, max_pos=64, num_blocks=2, block_size=8, seed=9, device="cpu")
    d["kv"][1:3] = 0
    d = to_device(d, cuda_device)
    dsv4_parity(d)
    ent = d["kv_cache"].view(-1, 584)[d["slot_mapping"][1]].cpu().numpy()
    assert np.all(ent[576:583] == 0) and np.all((ent[:448] & 0x7F) == 0)


def test_zero_tokens_is_a_no_op(cuda_device):
    d = wl.make_dsv4(0, 4, num_blocks=1, block_size=4, device=cuda_device)
    before = d["kv_cache"].clone()
    run_dsv4(d)
    torch.cuda.synchronize()
    assert torch.equal(before, d["kv_cache"])


def test_repeat_calls_are_deterministic(cuda_device):
    d = wl.make_dsv4(300, 8, max_pos=4096, num_blocks=16, block_size=64, seed=12,
                     device=cuda_device)
    d2 = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    run_dsv4(d)
    run_dsv4(d2)
    torch.cuda.synchronize()
    assert torch.equal(d["q"], d2["q"]) and torch.equal(d["kv_cache"], d2["kv_cache"])


DSV4_CONFIGS = list(range(5))


@pytest.mark.parametrize("config", DSV4_CONFIGS)
@pytest.mark.parametrize("shape", [(1, 1), (17, 3), (777, 5), (2048, 64)])
def test_every_launch_config(cuda_device, config, shape):
    """Each launch shape of the table against the oracle (forced)."""
    assert len(kvq.configs("dsv4")) == len(DSV4_CONFIGS)
    T, H = shape
    d = wl.make_dsv4(T, H, max_pos=131072, num_blocks=-(-2 * T // 16), block_size=16,
                     slots="distinct_skip2", seed=300 + config, device=cuda_device)
    with with_config("dsv4", config):
        dsv4_parity(d)


def _dsv4_run_config(d, config):
    q = d["q"].clone()
    cache = d["kv_cache"].clone()
    with with_config("dsv4", config):
        kvq.dsv4_qnorm_rope_kv_rope_quant_insert(q, d["kv"], d["eps"], d["q_weight"],
                                                 d["kv_weight"], d["cos_sin"], d["positions"],
                                                 d["slot_mapping"], cache)
    torch.cuda.synchronize()
    return q, cache


@pytest.mark.parametrize("shape", [(1, 1), (17, 3), (300, 7), (2048, 64), (513, 128)])
def test_launch_shapes_bit_identical(cuda_device, shape):
    """Every launch shape (one-shot, persistent) shares the row arithmetic: q
    and the whole cache come out as the same bytes."""
    T, H = shape
    d = wl.make_dsv4(T, H, max_pos=131072, num_blocks=-(-2 * T // 16), block_size=16,
                     slots="distinct_skip2", seed=400 + T + H, device=cuda_device)
    q_ref, c_ref = _dsv4_run_config(d, 4)
    assert not torch.equal(q_ref, d["q"])
    for config in DSV4_CONFIGS:
        q, c = _dsv4_run_config(d, config)
        assert torch.equal(q, q_ref) and torch.equal(c, c_ref), kvq.configs("dsv4")[config]


# ---- reading entries back (dsv4_kv_cache_gather) ---------------------------

def _gather_vs_oracle(cache_dev, slots):
    import oracle
    out = kvq.dsv4_kv_cache_gather(cache_dev, slots)
    torch.cuda.synchronize()
    want = oracle.dsv4_gather(wl.host(cache_dev), wl.host(slots))
    got = wl.bf16_bits(out)
    assert np.array_equal(got, want), f"{int((got != want).sum())} values differ"
    return got


@pytest.mark.parametrize("T,H", [(16, 64), (777, 3), (8192, 8)])
def test_gather_after_insert(cuda_device, T, H):
    """Insert on the GPU, read the entries back on the GPU: bit-exact against
    the oracle's reading of the same cache bytes, and within half an e4m3 step
    of the oracle's exact normalised values."""
    import oracle
    d = wl.make_dsv4(T, H, max_pos=131072, num_blocks=-(-2 * T // 64), block_size=64,
                     slots="distinct_skip2", seed=500 + T, device=cuda_device)
    q_in, cache_in = wl.bf16_bits(d["q"]), wl.host(d["kv_cache"]).copy()
    run_dsv4(d)
    slots = d["slot_mapping"]
    got = _gather_vs_oracle(d["kv_cache"], slots)
    res = oracle.dsv4(q_in, wl.bf16_bits(d["kv"]), d["eps"], wl.bf16_bits(d["q_weight"]),
                      wl.bf16_bits(d["kv_weight"]), wl.host(d["cos_sin"]), wl.host(d["positions"]),
                      wl.host(slots), cache_in, want_ref=True)
    m = wl.host(slots) >= 0
    vals = (got[m].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    n32 = res["kv_ref"][m].astype(np.float32).astype(np.float64)
    ent = wl.host(d["kv_cache"]).reshape(-1, 584)[wl.host(slots)[m]]
    scale = np.ldexp(1.0, ent[:, 576:583].astype(np.int64) - 127)
    err = np.abs(vals[:, :448] - n32[:, :448]).reshape(-1, 7, 64)
    bound = np.maximum(np.abs(n32[:, :448]).reshape(-1, 7, 64) * 2.0 ** -4,
                       scale[:, :, None] * 2.0 ** -10)
    assert np.all(err <= bound * (1 + 2.0 ** -10) + 1e-30)
    assert np.all(got[~m] == 0)


def test_gather_repeated_and_edge_slots(cuda_device):
    d = wl.make_dsv4(64, 2, max_pos=4096, num_blocks=2, block_size=64, seed=9, device=cuda_device)
    run_dsv4(d)
    slots = torch.tensor([0, 127, -1, 5, 5, 127, -1], dtype=torch.int64, device=cuda_device)
    _gather_vs_oracle(d["kv_cache"], slots)


def test_gather_hand_entry(cuda_device):
    """The hand-derived entry reads back as the block weights."""
    block_w = [1.0, 2.0, 4.0, 8.0, 0.5, 3.0, 5.0]
    codes = [0x78] * (5 * 64) + [0x7C] * 64 + [0x7A] * 64
    entry = np.array(codes + [0x80, 0x3F] * 64 + [119, 120, 121, 122, 118, 120, 121, 0], np.uint8)
    cache = np.full((1, 4, 584), 0xA5, np.uint8)
    cache.reshape(-1)[2 * 584:3 * 584] = entry
    out = kvq.dsv4_kv_cache_gather(torch.from_numpy(cache).to(cuda_device),
                                   torch.tensor([2], dtype=torch.int64, device=cuda_device))
    assert torch.equal(out[0].float().cpu(),
                       torch.tensor(np.repeat(block_w + [1.0], 64), dtype=torch.float32))


def test_cache_beyond_4_gib(cuda_device, parity_log):
    """A 4.9 GB cache (131072 blocks of 64 slots): every token maps to one of
    the last 4096 slots (entry offsets past 2^32 bytes, the very last slot
    included), through both launch shapes; then the entries are read back by
    the gather, bit-exact against the oracle's reading of the same bytes."""
    import oracle
    n = 131072 * 64
    assert (n - 4096) * 584 > 2**32
    for threshold in (SMALL_PATH, TILED_PATH):
        d = wl.make_dsv4(4096, 8, max_pos=131072, num_blocks=131072, block_size=64, seed=78,
                         device=cuda_device)
        g = torch.Generator(device=cuda_device).manual_seed(79)
        slots = n - 1 - torch.randperm(4096, generator=g, device=cuda_device)
        slots[[5, 2000]] = -1
        d["slot_mapping"] = slots
        with with_threshold(threshold):
            qrep, crep = dsv4_parity(d, sample=1024, seed=80)
        assert crep.exp_mismatch_ties == 0
        parity_log(qrep, crep)
        # read back: the entries at the sampled slots, compared through a
        # small host copy of exactly those entries
        read = torch.cat([slots[:64], torch.tensor([n - 1, -1], device=cuda_device)])
        out = kvq.dsv4_kv_cache_gather(d["kv_cache"], read)
        torch.cuda.synchronize()
        flat = d["kv_cache"].view(-1, 584)
        mapped = read >= 0
        small = torch.zeros((int(read.numel()), 584), dtype=torch.uint8, device=cuda_device)
        small[mapped] = flat[read[mapped]]
        local = torch.where(mapped, torch.arange(read.numel(), device=cuda_device), -1)
        want = oracle.dsv4_gather(wl.host(small).reshape(1, -1, 584), wl.host(local))
        assert np.array_equal(wl.bf16_bits(out), want)
        del d, slots, out, flat, small
        torch.cuda.empty_cache()


# ---- separate q output and CUDA-graph capture -------------------------------

@pytest.mark.parametrize("T,H,threshold", [(16, 64, None), (777, 5, TILED_PATH),
                                           (777, 5, SMALL_PATH), (4096, 64, None)])
def test_out_of_place_q(cuda_device, T, H, threshold):
    """q is read only, q_out receives the rows; against the oracle."""
    import oracle
    d = wl.make_dsv4(T, H, max_pos=131072, num_blocks=-(-2 * T // 64), block_size=64,
                     slots="distinct_skip2", seed=700 + T, device=cuda_device)
    q_before = d["q"].clone()
    cache_in = wl.host(d["kv_cache"]).copy()
    q_out = torch.full_like(d["q"], float("nan"))
    ctx = with_threshold(threshold) if threshold is not None else with_config("dsv4", -1)
    with ctx:
        kvq.dsv4_qnorm_rope_kv_rope_quant_insert(d["q"], d["kv"], d["eps"], d["q_weight"],
                                                 d["kv_weight"], d["cos_sin"], d["positions"],
                                                 d["slot_mapping"], d["kv_cache"], q_out=q_out)
    torch.cuda.synchronize()
    assert torch.equal(d["q"], q_before)
    res = oracle.dsv4(wl.bf16_bits(q_before), wl.bf16_bits(d["kv"]), d["eps"],
                      wl.bf16_bits(d["q_weight"]), wl.bf16_bits(d["kv_weight"]),
                      wl.host(d["cos_sin"]), wl.host(d["positions"]), wl.host(d["slot_mapping"]),
                      cache_in, want_ref=True)
    from parity import Bf16Report, compare_cache
    rep = Bf16Report()
    rep.add(wl.bf16_bits(q_out), res["q"], res["q_ref"], res["q_mag"])
    rep.check("q_out")
    compare_cache(wl.host(d["kv_cache"]), cache_in, wl.host(d["slot_mapping"]), res["kv_ref"],
                  res["kv_mag"], res["exp_margin"]).check("cache")


def _layer_inputs(dev, i, T_qk=17, T_ds=16):
    qk = wl.make_qk(T_qk, 16, 8, 8, theta=1e4, max_pos=4096, seed=800 + i, device=dev)
    ds = wl.make_dsv4(T_ds, 64, max_pos=65536, num_blocks=64, block_size=64,
                      slots="distinct_skip2", seed=900 + i, device=dev)
    return qk, ds


def _run_layer(qk, ds):
    kvq.fused_qk_norm_rope(qk["qkv"], 16, 8, 8, 128, qk["eps"], qk["q_weight"], qk["k_weight"],
                           qk["cos_sin"], True, qk["positions"])
    run_dsv4(ds)


def _clone(d):
    return {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


@pytest.mark.parametrize("large,staged,pdl", [(False, False, False), (True, False, False),
                                              (True, True, False), (False, False, True),
                                              (True, True, True)],
                         ids=["decode", "prefill", "prefill-staged", "decode-pdl",
                              "prefill-staged-pdl"])
def test_cuda_graph_capture_and_replay(cuda_device, large, staged, pdl):
    """Both operators recorded into one CUDA graph (several layers) and
    replayed twice give bit-identical results to the same calls run eagerly
    (also with the TMA-staged QK shape forced, and with programmatic
    dependent launch on)."""
    old = kvq.set_programmatic_launch(pdl)
    try:
        with with_config("qk", 7 if staged else -1):
            _graph_vs_eager(cuda_device, large)
    finally:
        kvq.set_programmatic_launch(old)


@pytest.mark.parametrize("staged", [False, True], ids=["tiles", "staged"])
def test_programmatic_launch_keeps_dependencies(cuda_device, staged):
    """With programmatic dependent launch on, kernels that read what the
    previous kernel on the stream wrote still see it: the packed-QKV operator
    applied twice to the same tensor, then an insert followed by a gather of
    the entries it wrote, give the bytes of ordinary launches."""
    qk = wl.make_qk(8192, 32, 8, 8, theta=1e6, max_pos=131072, seed=71, device=cuda_device)
    ds = wl.make_dsv4(2048, 64, max_pos=131072, num_blocks=64, block_size=64, seed=72,
                      device=cuda_device)

    def chain():
        a, b = _clone(qk), _clone(ds)
        for _ in range(3):
            kvq.fused_qk_norm_rope(a["qkv"], 32, 8, 8, 128, a["eps"], a["q_weight"],
                                   a["k_weight"], a["cos_sin"], True, a["positions"])
        run_dsv4(b)
        rows = kvq.dsv4_kv_cache_gather(b["kv_cache"], b["slot_mapping"])
        run_dsv4(b)
        torch.cuda.synchronize()
        return a["qkv"], b["q"], b["kv_cache"], rows

    with with_config("qk", 7 if staged else -1):
        ref = chain()
        old = kvq.set_programmatic_launch(True)
        try:
            got = chain()
        finally:
            kvq.set_programmatic_launch(old)
    for x, y in zip(ref, got):
        assert torch.equal(x, y)


def _graph_vs_eager(cuda_device, large):
    T_qk, T_ds = (4096, 2048) if large else (17, 16)
    layers = [_layer_inputs(cuda_device, i, T_qk, T_ds) for i in range(4)]
    eager = [(_clone(qk), _clone(ds)) for qk, ds in layers]
    graphed = [(_clone(qk), _clone(ds)) for qk, ds in layers]
    warm = [(_clone(qk), _clone(ds)) for qk, ds in layers]
    for qk, ds in warm:  # warm-up before capture (occupancy query, lazy init)
        _run_layer(qk, ds)
    torch.cuda.synchronize()
    for _ in range(2):
        for qk, ds in eager:
            _run_layer(qk, ds)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for qk, ds in graphed:
            _run_layer(qk, ds)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for (qe, de), (qg, dg) in zip(eager, graphed):
        assert torch.equal(qe["qkv"], qg["qkv"])
        assert torch.equal(de["q"], dg["q"]) and torch.equal(de["kv_cache"], dg["kv_cache"])

"""GPU parity of the decode path (router, top-k, gate/up GEMV + SwiGLU,
down GEMV + weighted combine, deduplicated small batches) against the CPU
oracle, through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from quantized_moe_expert_gemv_gb300 import binding, build, device, synth
from tests import parity
from tests.q4k_fixtures import dequant_test_blocks

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.load_library()
    oracle.build()


class Runner:
    """Plan + scratch + device layer for one shape; decode calls through the ABI."""

    def __init__(self, layer: synth.MoeLayer, max_n=binding.SI_MAX_DECODE_TOKENS):
        self.layer = layer
        self.shape = layer.shape
        self.dl = device.to_device(layer)
        self.plan = binding.si_moe_plan(device.desc_for(self.shape))
        self.scratch = device.alloc_scratch(self.plan, binding.SI_MODE_DECODE, max_n)

    def decode(self, x_bits: np.ndarray):
        s = self.shape
        n = x_bits.shape[0]
        x = device.tokens_to_device(x_bits)
        out = torch.empty((n, s.hidden), dtype=torch.float32, device="cuda")
        ids = torch.full((n, s.top_k), -1, dtype=torch.int32, device="cuda")
        w = torch.empty((n, s.top_k), dtype=torch.float32, device="cuda")
        counts = torch.full((s.n_experts,), -1, dtype=torch.int32, device="cuda")
        logits = torch.empty((n, s.n_experts), dtype=torch.float32, device="cuda")
        ro = binding.route_struct(topk_ids=ids, topk_w=w, expert_counts=counts, logits=logits)
        binding.si_moe_forward_decode(self.plan, self.dl.struct(), x, n, out, ro, self.scratch)
        assert binding.si_moe_read_status(self.plan, self.scratch) == binding.SI_OK
        return (out.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), counts.cpu().numpy(),
                logits.cpu().numpy())


def check_tokens(layer, x_bits, out, ids, w, sample=None):
    """Compare per-token GPU results with the oracle; return #near-tie tokens."""
    s = layer.shape
    rows = range(x_bits.shape[0]) if sample is None else sample
    o_ids, o_w, z64, margin = oracle.route_tokens(layer.router_w, x_bits, s.top_k,
                                                  bias=layer.router_bias, want_logits=True)
    near = 0
    for t in range(x_bits.shape[0]):
        if not parity.routing_ok(ids[t], o_ids[t], z64[t], margin[t], s.top_k):
            near += 1
            continue
        parity.same_by_id(ids[t], w[t], o_ids[t], o_w[t], atol=2e-6)
        assert abs(float(w[t].sum()) - 1.0) < 1e-5
    for t in rows:
        if set(ids[t].tolist()) != set(o_ids[t].tolist()):
            continue
        ref = oracle.moe_token(layer, x_bits[t])
        parity.assert_close(out[t], ref.out64, f"token {t}")
    return near


# ------------------------------------------------------------------ dequant
def test_debug_dequant_bit_exact_against_oracle():
    blocks = dequant_test_blocks()
    n = blocks.shape[0]
    ref = oracle.q4k_dequant(blocks)
    dev_blocks = torch.from_numpy(blocks).cuda()
    f32 = torch.empty(n * 256, dtype=torch.float32, device="cuda")
    bf = torch.empty(n * 256, dtype=torch.int16, device="cuda")
    binding.si_debug_q4k_dequant(dev_blocks, n, f32, bf)
    torch.cuda.synchronize()
    got = f32.cpu().numpy()
    finite = np.isfinite(ref)
    assert np.array_equal(got.view(np.uint32)[finite], ref.view(np.uint32)[finite])
    ref_bf = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(bf.cpu().numpy()[finite], ref_bf[finite])


def test_debug_dequant_qwen_layer_sample_bit_exact():
    layer_blocks = synth.q4k_random_blocks(synth.rng(1, 0, "gate"), 200_000)
    ref = oracle.q4k_dequant(layer_blocks)
    dev = torch.from_numpy(layer_blocks).cuda()
    f32 = torch.empty(ref.size, dtype=torch.float32, device="cuda")
    binding.si_debug_q4k_dequant(dev, layer_blocks.shape[0], f32, None)
    assert np.array_equal(f32.cpu().numpy().view(np.uint32), ref.view(np.uint32))


# -------------------------------------------------------------------- top-k
@pytest.mark.parametrize("E,k", [(8, 2), (128, 8), (256, 16), (16, 16), (5, 1), (33, 7)])
def test_debug_topk_bit_exact(E, k):
    g = np.random.default_rng(E * 100 + k)
    for trial in range(20):
        n = 1 + trial % 4
        if trial % 2:
            z = (g.integers(-4, 4, (n, E)) * 0.5).astype(np.float32)     # many exact ties
        else:
            z = g.normal(0, 1, (n, E)).astype(np.float32)
        desc = binding.make_desc(256, 256, E, k)
        ids = torch.full((n, k), -1, dtype=torch.int32, device="cuda")
        w = torch.empty((n, k), dtype=torch.float32, device="cuda")
        counts = torch.empty(E, dtype=torch.int32, device="cuda")
        binding.si_debug_topk(torch.from_numpy(z).cuda(), n, desc,
                              binding.route_struct(topk_ids=ids, topk_w=w, expert_counts=counts))
        ids_h, w_h = ids.cpu().numpy(), w.cpu().numpy()
        ref_counts = np.zeros(E, dtype=np.int64)
        for t in range(n):
            o = oracle.topk(z[t], k)
            assert np.array_equal(ids_h[t], o)
            np.testing.assert_allclose(w_h[t], oracle.renorm_weights(z[t].astype(np.float64), o),
                                       rtol=0, atol=2e-6)
            ref_counts[o] += 1
        assert np.array_equal(counts.cpu().numpy(), ref_counts)


# ------------------------------------------------------------ decode paths
@pytest.mark.parametrize("H,I,E,k", [(2048, 768, 128, 8), (256, 256, 8, 2), (2048, 768, 256, 16)])
def test_decode_single_token_router_ties_and_zero_rows(H, I, E, k):
    """Single-token routing with exact ties: identical router rows give
    bit-identical logits, and zero rows (of +0.0 or -0.0 weights) give zero
    logits; every tie goes to the lower expert index."""
    shape = synth.MoeShape(H, I, E, k)
    layer = synth.make_layer(shape, seed=41)
    g = np.random.default_rng(41)
    v = np.abs(g.normal(0, 0.02, H)).astype(np.float32)
    w_r = np.zeros((E, H), dtype=np.float32)
    w_r[: E // 8] = -0.0                      # the lowest rows are negative zeros
    top = [E - 1, E // 2, E // 4 + 1]         # three identical rows (in descending-id order)
    for e in top:
        w_r[e] = v
    if k > 3:
        w_r[E // 3] = 0.5 * v
        w_r[E - 2] = 0.5 * v
    layer.router_w = w_r
    layer.router_bias = None
    x = np.abs(synth.bf16_to_f32(synth.make_tokens(shape, seed=41, n_tokens=3))).astype(np.float32)
    x_bits = synth.bf16_bits(x)
    r = Runner(layer)
    for t in range(3):
        out, ids, w, counts, logits = r.decode(x_bits[t:t + 1])
        z = logits[0]
        assert z[0] == 0.0 and z[E // 8] == 0.0
        ref = oracle.topk(z, k)
        assert np.array_equal(ids[0], ref), (ids[0], ref)
        assert list(ids[0][:min(3, k)]) == sorted(top)[:min(3, k)]
        if k > 3:
            assert list(ids[0][3:5]) == sorted([E // 3, E - 2])
            assert list(ids[0][5:]) == list(range(k - 5)), "zero logits: lowest ids first"
        np.testing.assert_allclose(w[0], oracle.renorm_weights(z.astype(np.float64), ref), rtol=0, atol=2e-6)
        want = np.zeros(E, dtype=np.int32)
        want[ref] = 1
        assert np.array_equal(counts, want)
        o_ids, _, _, _ = oracle.route_tokens(layer.router_w, x_bits[t:t + 1], k, want_logits=True)
        assert np.array_equal(ids[0], o_ids[0])
        parity.assert_close(out[0], oracle.moe_token(layer, x_bits[t]).out64, f"token {t}")


def test_decode_tiny_layer_seed0():
    wl = synth.WORKLOADS["tiny"]
    layer = synth.make_layer(wl["shape"], seed=wl["seed"])
    x = synth.make_tokens(wl["shape"], seed=wl["seed"], n_tokens=33)
    r = Runner(layer)
    outs, idss, ws = [], [], []
    for t in range(x.shape[0]):
        out, ids, w, counts, logits = r.decode(x[t:t + 1])
        ref_counts = np.bincount(ids[0], minlength=layer.shape.n_experts)
        assert np.array_equal(counts, ref_counts)
        z_ref = oracle.router_logits(layer.router_w, x[t])
        np.testing.assert_allclose(logits[0], z_ref, rtol=0, atol=1e-5)
        outs.append(out[0]), idss.append(ids[0]), ws.append(w[0])
    near = check_tokens(layer, x, np.array(outs), np.array(idss), np.array(ws))
    assert near <= 1


def test_decode_qwen3_layer_routing_all_tokens_outputs_sampled():
    wl = synth.WORKLOADS["layer"]
    shape = wl["shape"]
    layer = synth.make_layer(shape, seed=wl["seed"])
    x = synth.make_tokens(shape, seed=wl["seed"], n_tokens=wl["n_tokens"])
    r = Runner(layer)
    outs = np.empty((x.shape[0], shape.hidden), np.float32)
    ids = np.empty((x.shape[0], shape.top_k), np.int32)
    ws = np.empty((x.shape[0], shape.top_k), np.float32)
    for t in range(x.shape[0]):
        o, i, w, c, _ = r.decode(x[t:t + 1])
        outs[t], ids[t], ws[t] = o[0], i[0], w[0]
        assert c.sum() == shape.top_k
    sample = list(range(0, x.shape[0], 97)) + [x.shape[0] - 1]
    near = check_tokens(layer, x, outs, ids, ws, sample=sample)
    assert near <= 3


@pytest.mark.parametrize("n", [2, 3, 4])
def test_decode_dedup_batches_match_per_token_oracle(n):
    wl = synth.WORKLOADS["dedup4"]
    shape, seed = wl["shape"], wl["seed"]
    bias = synth.dedup_router_bias(seed, synth.load_dedup_beta())
    layer = synth.make_layer(shape, seed=seed, router_bias=bias)
    x_all = synth.make_tokens(shape, seed, 4 * 6)
    r = Runner(layer)
    for step in range(3):
        x = x_all[4 * step: 4 * step + n]
        out, ids, w, counts, _ = r.decode(x)
        assert np.array_equal(counts, np.bincount(ids.reshape(-1), minlength=shape.n_experts))
        check_tokens(layer, x, out, ids, w)
        # one decode of n tokens == n decodes of one token
        for t in range(n):
            o1, i1, _, _, _ = r.decode(x[t:t + 1])
            assert np.array_equal(i1[0], ids[t])
            parity.assert_close(out[t], o1[0], "batched vs single")


@pytest.mark.parametrize("shape,n", [(synth.QWEN3_30B_A3B, 4), (synth.QWEN3_30B_A3B, 2), (synth.MoeShape(1024, 512, 64, 8), 3)])
def test_decode_batched_identical_tokens_reduce_to_one_token(shape, n):
    """n copies of one token: every distinct expert is chosen by all n tokens, so
    every unit of the multi-token kernel runs its full token loop (x, h and the
    down partials per token).  Each output must match the oracle and the
    single-token decode of the same token, with identical routing."""
    layer = synth.make_layer(shape, seed=41 + n)
    r = Runner(layer)
    assert binding.si_debug_decode_fused(r.plan, n) == 3
    x1 = synth.make_tokens(shape, seed=41 + n, n_tokens=1)
    x = np.repeat(x1, n, axis=0)
    out, ids, w, counts, _ = r.decode(x)
    o1, i1, w1, _, _ = r.decode(x1)
    assert np.array_equal(counts, np.bincount(ids.reshape(-1), minlength=shape.n_experts))
    assert sorted(set(counts.tolist()) - {0}) == [n]
    for t in range(n):
        assert np.array_equal(ids[t], i1[0])
        np.testing.assert_allclose(w[t], w1[0], rtol=0, atol=2e-6)
        parity.assert_close(out[t], o1[0], "batched copy vs single")
    check_tokens(layer, x, out, ids, w)


@pytest.mark.parametrize("H,I,E,k,n", [
    (256, 256, 8, 2, 1), (512, 768, 16, 4, 3), (768, 512, 4, 4, 2), (1024, 256, 32, 1, 4),
    (256, 1280, 6, 3, 1), (4096, 256, 8, 8, 2), (256, 256, 1, 1, 1), (2048, 768, 256, 16, 4),
    (1024, 512, 64, 8, 4), (2048, 256, 128, 4, 3), (1024, 256, 64, 2, 2),
])
def test_decode_shapes(H, I, E, k, n):
    shape = synth.MoeShape(H, I, E, k)
    layer = synth.make_layer(shape, seed=H + I + E + k)
    x = synth.make_tokens(shape, seed=7, n_tokens=n)
    out, ids, w, counts, _ = Runner(layer).decode(x)
    near = check_tokens(layer, x, out, ids, w)
    assert near == 0


def test_decode_identical_experts_any_routing():
    shape = synth.MoeShape(512, 512, 16, 4)
    layer = synth.make_layer(shape, seed=31)
    for name in ("w_gate", "w_up", "w_down"):
        arr = getattr(layer, name)
        arr[:] = arr[0]
    x = synth.make_tokens(shape, seed=31, n_tokens=4)
    out, _, _, _, _ = Runner(layer).decode(x)
    for t in range(4):
        xf = synth.bf16_to_f32(x[t]).astype(np.float64)
        _, y = oracle.expert_ffn(layer.w_gate[0], layer.w_up[0], layer.w_down[0], xf, 512, 512)
        parity.assert_close(out[t], y, "identical experts")


def test_decode_argument_errors():
    shape = synth.TINY
    layer = synth.make_layer(shape, seed=0)
    r = Runner(layer)
    x = device.tokens_to_device(synth.make_tokens(shape, 0, 2))
    out = torch.empty((2, shape.hidden), dtype=torch.float32, device="cuda")
    L = r.dl.struct()

    def call(xp, n, outp, scratch, nbytes=None):
        lib = binding.load_library()
        nb = nbytes if nbytes is not None else scratch.numel()
        import ctypes
        return lib.si_moe_forward_decode(r.plan.handle, ctypes.byref(L), xp, n, outp, None,
                                         scratch.data_ptr(), nb, torch.cuda.current_stream().cuda_stream)

    assert call(x.data_ptr() + 2, 1, out.data_ptr(), r.scratch) == binding.SI_ERR_MISALIGNED
    assert call(x.data_ptr(), 1, out.data_ptr() + 4, r.scratch) == binding.SI_ERR_MISALIGNED
    assert call(x.data_ptr(), 0, out.data_ptr(), r.scratch) == binding.SI_ERR_INVALID_ARG
    assert call(x.data_ptr(), 5, out.data_ptr(), r.scratch) == binding.SI_ERR_INVALID_ARG
    need = binding.si_moe_scratch_bytes(r.plan, binding.SI_MODE_DECODE, 2)
    assert call(x.data_ptr(), 2, out.data_ptr(), r.scratch, need - 1) == binding.SI_ERR_SCRATCH_TOO_SMALL
    assert call(x.data_ptr(), 2, out.data_ptr(), r.scratch, need) == binding.SI_OK
    assert binding.si_moe_read_status(r.plan, r.scratch) == binding.SI_OK


@pytest.mark.parametrize("workload,n", [("tiny", 1), ("layer", 1), ("dedup4", 4)])
def test_decode_host_buffers_match_the_oracle(workload, n):
    """si_moe_forward_decode_host: x from page-locked host memory, out back to
    it, the stream wait and the status read inside the call; then the same
    with pageable numpy buffers."""
    wl = synth.WORKLOADS[workload]
    shape, seed = wl["shape"], wl["seed"]
    bias = synth.dedup_router_bias(seed, synth.load_dedup_beta()) if workload == "dedup4" else None
    layer = synth.make_layer(shape, seed=seed, router_bias=bias)
    x = synth.make_tokens(shape, seed, 3 * n)
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(device.desc_for(shape))
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE_HOST, n)
    x_pin = torch.from_numpy(x.view(np.int16)).pin_memory()
    out_pin = torch.empty((n, shape.hidden), dtype=torch.float32).pin_memory()
    ids = torch.full((n, shape.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.empty((n, shape.top_k), dtype=torch.float32, device="cuda")
    ro = binding.route_struct(topk_ids=ids, topk_w=w)
    for step in range(3):
        out_pin.fill_(float("nan"))
        st = binding.si_moe_forward_decode_host(plan, dl.struct(), x_pin[step * n:(step + 1) * n], n, out_pin,
                                                ro, scratch)
        assert st == binding.SI_OK
        xs = x[step * n:(step + 1) * n]
        near = check_tokens(layer, xs, out_pin.numpy().copy(), ids.cpu().numpy(), w.cpu().numpy())
        assert near <= 1
    out_np = np.full((1, shape.hidden), np.nan, dtype=np.float32)
    x_np = np.ascontiguousarray(x[1:2])
    assert binding.si_moe_forward_decode_host(plan, dl.struct(), x_np, 1, out_np, ro, scratch) == binding.SI_OK
    check_tokens(layer, x_np, out_np, ids.cpu().numpy()[:1], w.cpu().numpy()[:1])


def test_decode_host_buffers_graph_cache_reuse_and_eviction():
    """The host-buffer call keeps a captured graph per (layer, route_out,
    scratch, n), at most four per plan: six scratch buffers in rotation make
    every call after the fourth evict and capture again, and a repeated key
    replays its graph with new host inputs."""
    shape = synth.TINY
    layer = synth.make_layer(shape, seed=0)
    dl = device.to_device(layer)
    x = synth.make_tokens(shape, 5, 12)
    plan = binding.si_moe_plan(device.desc_for(shape))
    scratches = [device.alloc_scratch(plan, binding.SI_MODE_DECODE_HOST, 2) for _ in range(6)]
    refs = [oracle.moe_token(layer, x[t]).out64 for t in range(x.shape[0])]
    for rep in range(2):
        for i, sc in enumerate(scratches):
            t = (2 * i + rep) % x.shape[0]
            out = np.full((1, shape.hidden), np.nan, dtype=np.float32)
            assert binding.si_moe_forward_decode_host(plan, dl.struct(), x[t:t + 1], 1, out, None, sc) == \
                binding.SI_OK
            parity.assert_close(out[0], refs[t], f"scratch {i}, token {t}")
    sc = scratches[0]
    for t in range(0, x.shape[0], 2):  # one key, new inputs every call, two tokens
        out = np.full((2, shape.hidden), np.nan, dtype=np.float32)
        assert binding.si_moe_forward_decode_host(plan, dl.struct(), x[t:t + 2], 2, out, None, sc) == binding.SI_OK
        for j in range(2):
            parity.assert_close(out[j], refs[t + j], f"token {t + j}")


def test_decode_host_buffers_argument_errors_and_timeout(monkeypatch):
    shape = synth.TINY
    layer = synth.make_layer(shape, seed=0)
    dl = device.to_device(layer)
    x = synth.make_tokens(shape, 0, 1)
    out = np.full((1, shape.hidden), np.nan, dtype=np.float32)
    plan = binding.si_moe_plan(device.desc_for(shape))
    small = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)  # no room for the staging of x and out
    st = binding.si_moe_forward_decode_host(plan, dl.struct(), x, 1, out, None, small, raw_status=True)
    assert st == binding.SI_ERR_SCRATCH_TOO_SMALL and np.isnan(out).all()
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE_HOST, 1)
    assert binding.si_moe_forward_decode_host(plan, dl.struct(), None, 1, out, None, scratch,
                                              raw_status=True) == binding.SI_ERR_INVALID_ARG
    assert binding.si_moe_forward_decode_host(plan, dl.struct(), x, 5, out, None, scratch,
                                              raw_status=True) == binding.SI_ERR_INVALID_ARG
    assert np.isnan(out).all()
    # a wait that runs out is returned by the call itself, and cleared
    monkeypatch.setenv("SI_FAULT_WAIT_BUDGET", "0")
    plan0 = binding.si_moe_plan(device.desc_for(shape))
    monkeypatch.delenv("SI_FAULT_WAIT_BUDGET")
    assert binding.si_moe_forward_decode_host(plan0, dl.struct(), x, 1, out, None, scratch,
                                              raw_status=True) == binding.SI_ERR_TIMEOUT
    assert binding.si_moe_read_status(plan0, scratch) == binding.SI_OK
    binding.si_moe_scratch_init(plan, scratch)
    assert binding.si_moe_forward_decode_host(plan, dl.struct(), x, 1, out, None, scratch) == binding.SI_OK
    parity.assert_close(out[0], oracle.moe_token(layer, x[0]).out64, "host buffers after a timeout")


def test_decode_in_cuda_graph_matches_eager():
    wl = synth.WORKLOADS["layer"]
    shape = wl["shape"]
    layer = synth.make_layer(shape, seed=wl["seed"])
    r = Runner(layer)
    xb = synth.make_tokens(shape, seed=wl["seed"], n_tokens=8)
    x = device.tokens_to_device(xb)
    out = torch.zeros((8, shape.hidden), dtype=torch.float32, device="cuda")
    L = r.dl.struct()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for t in range(8):   # warm-up outside capture
            binding.si_moe_forward_decode(r.plan, L, x[t], 1, out[t], None, r.scratch, stream=s)
    s.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for t in range(8):
            binding.si_moe_forward_decode(r.plan, L, x[t], 1, out[t], None, r.scratch, stream=s)
    g.replay()
    torch.cuda.synchronize()
    # the single-token path combines the top-k slots with float reductions: equal up to rounding order
    for t in range(8):
        parity.assert_close(out[t].cpu().numpy(), eager[t].cpu().numpy(), "graph replay vs eager")


def test_fused_path_is_taken_for_the_qwen3_shape():
    plan = binding.si_moe_plan(device.desc_for(synth.QWEN3_30B_A3B))
    assert binding.si_debug_decode_fused(plan, 1) == 2            # cluster kernel
    info = binding.si_debug_plan_info(plan)
    assert info["cluster_ok"] == 1 and 2 <= info["cluster_size"] <= 8
    assert info["clusters_resident"] >= info["clusters_needed"] == 24   # one wave
    for n in range(2, binding.SI_MAX_DECODE_TOKENS + 1):
        assert binding.si_debug_decode_fused(plan, n) == 3        # cluster kernel over the distinct experts
    plan_h768 = binding.si_moe_plan(binding.make_desc(768, 512, 4, 4))
    assert binding.si_debug_decode_fused(plan_h768, 1) == 0


@pytest.mark.parametrize("n,prenorm,shape", [(1, False, synth.TINY), (2, False, synth.MoeShape(1024, 256, 64, 4)),
                                             (2, True, synth.TINY)])
def test_bounded_wait_timeout_is_reported_and_the_context_survives(monkeypatch, n, prenorm, shape):
    """A wait budget of 0 cycles makes every device-side wait of the expert
    kernel (cluster kernel for n = 1, the cluster kernel over the distinct
    experts for n = 2, the grid-synchronised kernel for n = 2 in a pre-normed
    block) give up at once: the kernel must record SI_ERR_TIMEOUT, let its
    copies land, and return; the next call on a fresh scratch must be right."""
    layer = synth.make_layer(shape, seed=0)
    if prenorm:
        layer.norm_weight = synth.make_norm_weight(shape, seed=0)
        layer.norm_eps = 1e-6
    dl = device.to_device(layer)
    x_bits = synth.make_tokens(shape, seed=0, n_tokens=n)
    x = device.tokens_to_device(x_bits)
    monkeypatch.setenv("SI_FAULT_WAIT_BUDGET", "0")
    plan0 = binding.si_moe_plan(device.desc_for(shape))
    monkeypatch.delenv("SI_FAULT_WAIT_BUDGET")
    assert binding.si_debug_decode_fused(plan0, n) == (2 if n == 1 else 3 if not prenorm else 1)
    scratch = device.alloc_scratch(plan0, binding.SI_MODE_DECODE, n)
    out = torch.zeros((n, shape.hidden), dtype=torch.float32, device="cuda")
    binding.si_moe_forward_decode(plan0, dl.struct(), x, n, out, None, scratch)
    assert binding.si_moe_read_status(plan0, scratch) == binding.SI_ERR_TIMEOUT
    assert binding.si_moe_read_status(plan0, scratch) == binding.SI_OK   # reading clears it
    # a normal plan on a re-initialised scratch gives the right answer
    plan = binding.si_moe_plan(device.desc_for(shape))
    binding.si_moe_scratch_init(plan, scratch)
    binding.si_moe_forward_decode(plan, dl.struct(), x, n, out, None, scratch)
    assert binding.si_moe_read_status(plan, scratch) == binding.SI_OK
    for t in range(n):
        if prenorm:
            ref = oracle.moe_token_prenorm(layer, x_bits[t], layer.norm_weight, layer.norm_eps)
        else:
            ref = oracle.moe_token(layer, x_bits[t])
        parity.assert_close(out.cpu().numpy()[t], ref.out64, "after timeout")


def test_fault_budget_env_polarity(monkeypatch):
    """The budget override is on only when set to a decimal number."""
    for val in ("", "abc", "-5", "12x"):
        monkeypatch.setenv("SI_FAULT_WAIT_BUDGET", val)
        plan = binding.si_moe_plan(device.desc_for(synth.TINY))
        shape = synth.TINY
        layer = synth.make_layer(shape, seed=0)
        r = Runner(layer)
        r.plan = plan
        out, ids, w, counts, _ = r.decode(synth.make_tokens(shape, 0, 1))   # asserts SI_OK status

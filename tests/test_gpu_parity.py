"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every workload shape runs through the same entry points the bench times
(ep_route -> ep_dispatch -> ep_combine on one stream, and ep_route_dispatch
in each of its forms). Every output is compared in full, at T=131072, H=8192
too (there one rank block or token range at a time). Tolerances are stated in
tests/parity.py.
"""
import numpy as np
import pytest
import torch

from parity import assert_combine_close, assert_weights_close, bf16_to_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from combine_warp_top_fp32_b300 import binding

    return binding


def _bits(t):
    from combine_warp_top_fp32_b300.workloads import bf16_bits

    return bf16_bits(t)


def _run_path(ep, cfg, logits, x, expert_out):
    buf = ep.EpBuffers.allocate(cfg)
    buf.step(logits, x, expert_out)
    torch.cuda.synchronize()
    assert ep.ep_get_error(buf.ws) == ep.EP_OK
    return buf


_OUTPUTS = ("topk_idx", "topk_w", "slot_row", "expert_counts", "expert_raw", "expert_off", "rank_off", "n_dropped")


def _assert_fused_matches(ep, cfg, ref, logits, x):
    """ep_route_dispatch writes bit-for-bit what ep_route + ep_dispatch wrote,
    in each of its forms: the library's choice, the single cooperative launch
    (where the shape allows it) and the kernel chain."""
    try:
        for form in (ep.EP_FORM_AUTO, ep.EP_FORM_SINGLE, ep.EP_FORM_CHAIN):
            ep.ep_debug_set(ep.EP_DEBUG_ROUTE_DISPATCH_FORM, form)
            fused = ep.EpBuffers.allocate(cfg)
            fused.route_dispatch(logits, x)
            torch.cuda.synchronize()
            assert ep.ep_get_error(fused.ws) == ep.EP_OK
            for name in _OUTPUTS:
                assert torch.equal(getattr(ref, name), getattr(fused, name)), (form, name)
            N = int(ref.rank_off[-1].item())
            assert torch.equal(ref.row_slot[:N], fused.row_slot[:N]), form
            assert torch.equal(ref.payload[:N].view(torch.uint8), fused.payload[:N].view(torch.uint8)), form
            if ref.scales is not None:
                assert torch.equal(ref.scales[:N], fused.scales[:N]), form
            del fused
    finally:
        ep.ep_debug_set(ep.EP_DEBUG_ROUTE_DISPATCH_FORM, ep.EP_FORM_AUTO)


def _check_layout(buf, lay, N):
    np.testing.assert_array_equal(buf.expert_counts.cpu().numpy(), lay["expert_counts"])
    np.testing.assert_array_equal(buf.expert_raw.cpu().numpy(), lay["expert_raw"])
    np.testing.assert_array_equal(buf.expert_off.cpu().numpy(), lay["expert_off"])
    np.testing.assert_array_equal(buf.rank_off.cpu().numpy(), lay["rank_off"])
    assert int(buf.n_dropped.item()) == lay["n_dropped"]
    np.testing.assert_array_equal(buf.slot_row.cpu().numpy(), lay["slot_row"])
    np.testing.assert_array_equal(buf.row_slot[:N].cpu().numpy(), lay["row_slot"])


def _full_parity(ep, orc, w, payload, renormalize=False, device_gen="cuda"):
    from combine_warp_top_fp32_b300 import workloads

    w = w.replace(renormalize=renormalize)
    cfg = ep.config_from_workload(w, payload=payload)
    d = workloads.generate(w, device=device_gen)
    logits, x, eo = (d[n].cuda() for n in ("logits", "x", "expert_out"))
    buf = _run_path(ep, cfg, logits, x, eo)
    _assert_fused_matches(ep, cfg, buf, logits, x)

    logits_h = logits.cpu().numpy()
    x_bits = _bits(x)
    eo_bits = _bits(eo)
    # route: indices bit-exact, weights within 1e-6 relative
    idx, wts = orc.route(logits_h, w.k, renormalize)
    np.testing.assert_array_equal(buf.topk_idx.cpu().numpy(), idx)
    worst_w = assert_weights_close(buf.topk_w.cpu().numpy(), wts)
    # counts, offsets, permutation: bit-exact
    lay = orc.layout(idx, w.E, w.R, w.capacity_factor)
    N = lay["N"]
    _check_layout(buf, lay, N)
    # payload: bit-exact bytes (bf16) or codes + scales (int8, FP8 E4M3)
    pl, sc = orc.payload(x_bits, lay["row_slot"], w.k, payload)
    if payload != ep.EP_PAYLOAD_BF16:
        np.testing.assert_array_equal(buf.payload[:N].cpu().numpy(), pl)
        np.testing.assert_array_equal(buf.scales[:N].cpu().numpy(), sc)
    else:
        np.testing.assert_array_equal(_bits(buf.payload[:N]), pl)
    # combine through the whole path
    y_orc = orc.combine(eo_bits, None, lay["slot_row"], wts, w.T, w.k)
    eo_f = lambda rows: bf16_to_f32(eo_bits[rows]).astype(np.float64)
    stats = assert_combine_close(_bits(buf.y), y_orc, wts, lay["slot_row"], eo_f, w.k)
    # combine alone on identical inputs: bit-exact
    slot_row_d = torch.from_numpy(lay["slot_row"]).cuda()
    w_d = torch.from_numpy(wts).cuda()
    y2 = torch.empty_like(buf.y)
    ep.ep_combine(cfg, eo, None, ep.EP_PAYLOAD_BF16, slot_row_d, w_d, y2, buf.ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(y2), y_orc)
    return dict(N=N, dropped=lay["n_dropped"], worst_w_rel=worst_w, **stats)


CASES = [("tiny", 0), ("decode-latency", 1), ("prefill-mid", 0), ("prefill-mid", 1), ("capacity", 1),
         # FP8 E4M3 and int4 per-token payloads (the lower-precision extension)
         ("decode-latency", 2), ("prefill-mid", 2), ("capacity", 2),
         ("decode-latency", 3), ("prefill-mid", 3), ("capacity", 3)]


@pytest.mark.parametrize("name,payload", CASES)
def test_workload_parity(ep, orc, name, payload):
    from combine_warp_top_fp32_b300 import workloads

    info = _full_parity(ep, orc, workloads.WORKLOADS[name], payload)
    print(name, payload, info)
    if name == "capacity":
        assert info["dropped"] > 0  # the cap binds on this skewed workload


@pytest.mark.parametrize("name", ["tiny", "prefill-mid"])
def test_workload_parity_renormalized(ep, orc, name):
    from combine_warp_top_fp32_b300 import workloads

    _full_parity(ep, orc, workloads.WORKLOADS[name], 0, renormalize=True)


@pytest.mark.parametrize("payload", [0, 1, 2, 3])
def test_large_parity_full(ep, orc, payload):
    """T=131072, H=8192, E=256, k=8 at full size, in the bench's launch
    configuration, compared in full with the oracle: routing and all layout
    metadata at once; every payload row and scale one rank block at a time
    (131,072 rows each); every combined token one 8192-token range at a time
    (the expert-output rows each range needs are gathered to the host)."""
    from combine_warp_top_fp32_b300 import workloads

    w = workloads.WORKLOADS["large"]
    cfg = ep.config_from_workload(w, payload=payload)
    d = workloads.generate(w, device="cuda")
    logits, x, eo = d["logits"], d["x"], d["expert_out"]
    buf = _run_path(ep, cfg, logits, x, eo)
    _assert_fused_matches(ep, cfg, buf, logits, x)
    idx, wts = orc.route(logits.cpu().numpy(), w.k)
    np.testing.assert_array_equal(buf.topk_idx.cpu().numpy(), idx)
    assert_weights_close(buf.topk_w.cpu().numpy(), wts)
    lay = orc.layout(idx, w.E, w.R, w.capacity_factor)
    N = lay["N"]
    assert N == w.T * w.k
    _check_layout(buf, lay, N)

    # payload and scales, per rank block: the count of mismatching rows must be 0 in every block
    x_bits = _bits(x)
    roff = lay["rank_off"]
    bad_rows = []
    for r in range(w.R):
        r0, r1 = int(roff[r]), int(roff[r + 1])
        pl, sc = orc.payload(x_bits, lay["row_slot"][r0:r1], w.k, payload)
        got = buf.payload[r0:r1]
        got = _bits(got) if payload == ep.EP_PAYLOAD_BF16 else got.cpu().numpy()
        bad = np.any(got.reshape(r1 - r0, -1) != pl.reshape(r1 - r0, -1), axis=1)
        if sc is not None:
            bad |= buf.scales[r0:r1].cpu().numpy().view(np.uint32) != sc.view(np.uint32)
        bad_rows.append(int(np.count_nonzero(bad)))
        del pl, sc, got
    print("large payload", payload, "mismatching rows per rank block", bad_rows)
    assert bad_rows == [0] * w.R
    del x_bits

    # every combined token, per range of tokens
    sr_all = lay["slot_row"].reshape(w.T, w.k)
    beyond = 0
    for t0 in range(0, w.T, 8192):
        t1 = min(w.T, t0 + 8192)
        sr = sr_all[t0:t1]
        need = np.unique(sr[sr >= 0])
        eo_sub = _bits(eo.index_select(0, torch.from_numpy(need).long().cuda()))
        remap = np.full(N, -1, np.int64)
        remap[need] = np.arange(need.size)
        sr_sub = np.where(sr >= 0, remap[np.maximum(sr, 0)], -1).astype(np.int32)
        w_sub = wts[t0:t1]
        y_orc = orc.combine(eo_sub, None, sr_sub, w_sub, t1 - t0, w.k)
        y_gpu = _bits(buf.y[t0:t1])
        eo_f = lambda rr, e=eo_sub: bf16_to_f32(e[rr]).astype(np.float64)
        beyond += assert_combine_close(y_gpu, y_orc, w_sub, sr_sub, eo_f, w.k)["beyond_1ulp"]
        del eo_sub, y_orc, y_gpu
    print("large combine", payload, "elements beyond 1 bf16 ulp (cancellation bound)", beyond)


# ----------------------------------------------------------------------------
# edge cases: ragged tiles, extreme sizes, degenerate routing
# ----------------------------------------------------------------------------
EDGE = [
    # T, H, E, k, R, cf, payload, renorm, note
    (1, 16, 1, 1, 1, 0.0, 0, 0, "one token, one expert, minimum H"),
    (5, 16, 3, 2, 1, 0.0, 1, 0, "int8 at minimum H: one 16-element group"),
    (700, 48, 6, 3, 3, 0.0, 1, 0, "int8 with an odd number of 16-element groups"),
    (5, 16, 3, 2, 1, 0.0, 2, 0, "FP8 at minimum H"),
    (1000, 64, 8, 2, 2, 0.5, 2, 1, "FP8 with drops and a ragged last tile"),
    (777, 16384, 4, 2, 2, 0.0, 2, 0, "FP8 at maximum H"),
    (5, 32, 3, 2, 1, 0.0, 3, 0, "int4 at its minimum H"),
    (1000, 96, 8, 2, 2, 0.5, 3, 1, "int4 with drops and a ragged last tile"),
    (777, 16384, 4, 2, 2, 0.0, 3, 0, "int4 at maximum H"),
    (1000, 64, 8, 2, 2, 0.0, 1, 0, "ragged last tile"),
    (2500, 48, 6, 3, 3, 0.0, 0, 1, "E not a power of two, two ragged tiles"),
    (777, 16384, 4, 2, 2, 0.0, 1, 0, "maximum H"),
    (300, 32, 1024, 32, 8, 0.0, 1, 1, "maximum E and k"),
    (513, 32, 160, 5, 160, 0.0, 0, 0, "E = R: one expert per rank, non-pow2 values per lane"),
    (400, 64, 16, 16, 4, 0.0, 0, 0, "k = E: every expert"),
    (3000, 128, 32, 4, 4, 0.25, 1, 0, "heavy capacity drops"),
    (2048, 256, 64, 6, 8, 1.0, 0, 1, "capacity factor 1.0, bf16"),
    (40000, 16, 512, 4, 8, 1.0, 1, 0, "many experts x tiles (80,384 tile counts)"),
    (256, 64, 256, 8, 8, 0.5, 1, 1, "largest batch laid out by one cluster (8 tiles), E=256, drops"),
    (257, 64, 256, 8, 8, 0.0, 0, 0, "one token past the cluster layout"),
    (200, 32, 257, 3, 1, 0.0, 1, 0, "E=257: past the cluster layout's expert limit"),
    (100, 32, 160, 5, 8, 0.3, 0, 0, "cluster layout, 5 values per lane, ragged tile, drops"),
    (250, 64, 64, 6, 8, 0.0, 2, 0, "cluster layout, two tokens per warp in flight"),
    (33, 48, 3, 3, 3, 0.0, 1, 1, "cluster layout of two tiles, one token in the second"),
    (200, 32, 64, 32, 4, 0.5, 1, 1, "cluster layout at the maximum k = 32, drops"),
    (160, 64, 256, 1, 256, 0.0, 3, 0, "cluster layout, k = 1, one expert per rank, int4"),
]


@pytest.mark.parametrize("T,H,E,k,R,cf,payload,renorm,note", EDGE, ids=[e[-1] for e in EDGE])
def test_edge_case_parity(ep, orc, T, H, E, k, R, cf, payload, renorm, note):
    from combine_warp_top_fp32_b300 import workloads

    w = workloads.Workload("edge", T=T, H=H, E=E, k=k, R=R, capacity_factor=cf, payloads=(payload,), seed=T + E,
                           sigma_bias=1.0)
    info = _full_parity(ep, orc, w, payload, renormalize=bool(renorm), device_gen="cpu")
    if cf == 0.25:
        assert info["dropped"] > 0


def test_all_ties_pick_lowest_ids(ep, orc):
    cfg = ep.make_config(64, 32, 16, 4, 4)
    logits = torch.zeros(64, 16, device="cuda")
    logits[::2] = -0.0  # -0 and +0 tie
    buf = ep.EpBuffers.allocate(cfg)
    buf.route(logits)
    torch.cuda.synchronize()
    assert np.all(buf.topk_idx.cpu().numpy() == np.arange(4))
    np.testing.assert_allclose(buf.topk_w.cpu().numpy(), 1.0 / 16, rtol=1e-6)


def test_empty_batch_fused(ep):
    cfg = ep.make_config(0, 64, 8, 2, 2, payload=ep.EP_PAYLOAD_INT8)
    buf = ep.EpBuffers.allocate(cfg)
    buf.expert_off.fill_(7)
    buf.rank_off.fill_(7)
    buf.n_dropped.fill_(7)
    buf.route_dispatch(torch.empty(0, 8, device="cuda"), torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert buf.expert_off.cpu().tolist() == [0] * 9
    assert buf.rank_off.cpu().tolist() == [0] * 3
    assert buf.n_dropped.item() == 0
    assert ep.ep_get_error(buf.ws) == ep.EP_OK


def test_empty_batch(ep):
    cfg = ep.make_config(0, 64, 8, 2, 2, payload=ep.EP_PAYLOAD_INT8)
    buf = ep.EpBuffers.allocate(cfg)
    buf.expert_off.fill_(7)
    buf.rank_off.fill_(7)
    buf.n_dropped.fill_(7)
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    buf.step(torch.empty(0, 8, device="cuda"), x, torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert buf.expert_off.cpu().tolist() == [0] * 9
    assert buf.rank_off.cpu().tolist() == [0] * 3
    assert buf.n_dropped.item() == 0
    assert ep.ep_get_error(buf.ws) == ep.EP_OK


@pytest.mark.parametrize("fmt", ["int8", "fp8", "int4"])
@pytest.mark.parametrize("shape", ["prefill-mid", "wide", "many-slots", "many-slots-drops", "short"])
def test_coded_return_path(ep, orc, shape, fmt):
    """Expert outputs coded per row (ep_quantize_rows / _fp8 / _int4) then
    combined from the codes. prefill-mid: 2 KB rows; wide: 8 KB rows, with
    drops; many-slots: k = 16, every slot kept (more than 8 kept slots: the
    sum runs in groups of 8 with the accumulators carried); many-slots-drops:
    k = 12 with heavy drops (0 to 12 kept slots per token); short: T = 37, so
    each token's row is cut into slices."""
    from combine_warp_top_fp32_b300 import workloads

    fp8, int4 = fmt == "fp8", fmt == "int4"
    w = workloads.WORKLOADS["prefill-mid"]
    if shape == "wide":
        w = w.replace(T=1500, H=8192, capacity_factor=1.0, seed=9)
    elif shape == "many-slots":
        w = w.replace(T=700, H=1024, E=64, k=16, capacity_factor=0.0, seed=11)
    elif shape == "many-slots-drops":
        w = w.replace(T=900, H=2048, E=32, k=12, capacity_factor=0.5, seed=12)
    elif shape == "short":
        w = w.replace(T=37, H=4096, E=64, k=6, capacity_factor=0.0, seed=13)
    kind = {"int8": ep.EP_PAYLOAD_INT8, "fp8": ep.EP_PAYLOAD_FP8, "int4": ep.EP_PAYLOAD_INT4}[fmt]
    cfg = ep.config_from_workload(w, payload=kind)
    d = workloads.generate(w, device="cuda")
    rows = w.max_rows()
    q = torch.empty(rows, w.H // 2 if int4 else w.H, dtype=torch.int8 if fmt == "int8" else torch.uint8,
                    device="cuda")
    s = torch.empty(rows, dtype=torch.float32, device="cuda")
    quant = {"int8": ep.ep_quantize_rows, "fp8": ep.ep_quantize_rows_fp8, "int4": ep.ep_quantize_rows_int4}[fmt]
    quant(d["expert_out"], q, s)
    torch.cuda.synchronize()
    q_o, s_o = orc.quantize_rows(_bits(d["expert_out"]), fp8=fp8, int4=int4)
    np.testing.assert_array_equal(q.cpu().numpy(), q_o)
    np.testing.assert_array_equal(s.cpu().numpy(), s_o)
    idx, wts = orc.route(d["logits"].cpu().numpy(), w.k)
    lay = orc.layout(idx, w.E, w.R, w.capacity_factor)
    y_orc = orc.combine(q_o, s_o, lay["slot_row"], wts, w.T, w.k, int4=int4)
    buf = ep.EpBuffers.allocate(cfg)
    y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    ep.ep_combine(cfg, q, s, kind, torch.from_numpy(lay["slot_row"]).cuda(), torch.from_numpy(wts).cuda(), y,
                  buf.ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(y), y_orc)


def test_combine_slot_order_and_fma(ep, orc):
    """The two combine pins of the oracle on the GPU: token 0 sums 2^24, 1,
    -2^24 in slot order (0 in fp32 with ties to even, 1 in any other order);
    token 1 adds w1*v1 to -fl(w1*v1), which only a fused multiply-add leaves
    as the nonzero residual."""
    H, k, T = 16, 3, 2
    w1 = np.float32(1.0 + 2.0**-20 + 2.0**-23)
    v1 = np.float32(1.0 + 2.0**-7)
    P = np.float32(w1 * v1)
    vals = np.array([2.0**24, 1.0, -(2.0**24), -1.0, v1], np.float32)
    eo = (np.repeat(vals[:, None], H, axis=1).view(np.uint32) >> 16).astype(np.uint16)  # exact in bf16
    slot_row = np.array([0, 1, 2, 3, 4, -1], np.int32)
    w = np.array([1.0, 1.0, 1.0, P, w1, 0.5], np.float32)
    y_orc = orc.combine(eo, None, slot_row, w, T, k)
    cfg = ep.make_config(T, H, 8, k, 1)
    buf = ep.EpBuffers.allocate(cfg)
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    ep.ep_combine(cfg, torch.from_numpy(eo.view(np.int16)).cuda().view(torch.bfloat16), None, ep.EP_PAYLOAD_BF16,
                  torch.from_numpy(slot_row).cuda(), torch.from_numpy(w).cuda(), y, buf.ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(y), y_orc)
    assert np.all(bf16_to_f32(y_orc[0]) == 0.0) and np.all(bf16_to_f32(y_orc[1]) != 0.0)


@pytest.mark.parametrize("fmt", ["int8", "fp8", "int4"])
def test_combine_decodes_every_code(ep, orc, fmt):
    """Every code value (256 int8 bytes, 254 non-NaN E4M3 bytes, 16 nibbles in
    every position) widened by the combine and summed over two slots, against
    the oracle's combine on the same codes, bit for bit. Scales span normal,
    tiny (subnormal products) and large values."""
    T, k, E = 8, 2, 8
    int4 = fmt == "int4"
    H = 512 if int4 else 256
    kind = {"int8": ep.EP_PAYLOAD_INT8, "fp8": ep.EP_PAYLOAD_FP8, "int4": ep.EP_PAYLOAD_INT4}[fmt]
    rng = np.random.default_rng(17)
    rows = T * k
    codes = np.stack([rng.permutation(256) for _ in range(rows)]).astype(np.uint8)  # every byte in every row
    if fmt == "fp8":
        codes[(codes & 0x7F) == 0x7F] ^= 1  # E4M3 NaN codes are never written: 0x7F -> 0x7E, 0xFF -> 0xFE
    q_np = codes.view(np.int8) if fmt == "int8" else codes
    s_np = np.array([1.0, 0.37, 3.1e-3, 2.0 ** -120, 1.0e-38, 5.5e3, 0.0, 1.7e30] * 2, np.float32)
    w_np = rng.uniform(0.05, 1.0, (T, k)).astype(np.float32)
    slot_row = rng.permutation(rows).astype(np.int32).reshape(T, k)
    slot_row[3, 1] = -1  # a dropped slot
    y_orc = orc.combine(q_np, s_np, slot_row, w_np, T, k, int4=int4)
    cfg = ep.make_config(T, H, E, k, 1, payload=kind)
    buf = ep.EpBuffers.allocate(cfg)
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    ep.ep_combine(cfg, torch.from_numpy(q_np).cuda(), torch.from_numpy(s_np).cuda(), kind,
                  torch.from_numpy(slot_row).cuda(), torch.from_numpy(w_np).cuda(), y, buf.ws)
    torch.cuda.synchronize()
    assert ep.ep_get_error(buf.ws) == ep.EP_OK
    np.testing.assert_array_equal(_bits(y), y_orc)


@pytest.mark.parametrize("payload", [0, 1, 2, 3])
def test_identity_experts_round_trip(ep, payload):
    """combine(dispatch(x)) with identity experts and renormalised weights gives x back."""
    T, H, E, k, R = 2048, 512, 32, 4, 4
    cfg = ep.make_config(T, H, E, k, R, renormalize=True, payload=payload)
    g = torch.Generator(device="cuda").manual_seed(5)
    logits = torch.randn(T, E, device="cuda", generator=g)
    x = torch.randn(T, H, device="cuda", generator=g).to(torch.bfloat16)
    buf = ep.EpBuffers.allocate(cfg)
    buf.route(logits)
    buf.dispatch(x)
    buf.combine(buf.payload, buf.scales)
    torch.cuda.synchronize()
    xf = x.float().cpu().numpy().astype(np.float64)
    yf = buf.y.float().cpu().numpy().astype(np.float64)
    from parity import bf16_ulp

    if payload == 0:
        assert np.all(np.abs(yf - xf) <= bf16_ulp(xf))
    else:
        s_tok = np.zeros(T)
        rs = buf.row_slot.cpu().numpy()
        s_tok[rs // k] = buf.scales.cpu().numpy()
        if payload in (1, 3):  # int8, int4: half a code step
            bound = (s_tok / 2)[:, None] * 1.0001
        else:  # E4M3: 2^-4 relative above 2^-6 * scale, 2^-10 * scale below
            bound = np.maximum(np.abs(xf) * 2.0 ** -4, (s_tok * 2.0 ** -10)[:, None]) * 1.0001
        assert np.all(np.abs(yf - xf) <= bound + bf16_ulp(xf))


def test_deterministic_bytes(ep):
    from combine_warp_top_fp32_b300 import workloads

    w = workloads.WORKLOADS["prefill-mid"]
    cfg = ep.config_from_workload(w, payload=ep.EP_PAYLOAD_INT8)
    d = workloads.generate(w, device="cuda")
    outs = []
    for _ in range(2):
        buf = _run_path(ep, cfg, d["logits"], d["x"], d["expert_out"])
        outs.append([t.clone() for t in (buf.topk_idx, buf.topk_w, buf.payload, buf.scales, buf.slot_row, buf.y)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_wait_and_work_words_return_to_zero(ep):
    """Every call leaves the workspace's words where the next call expects
    them: after capacity steps the single launch's arrival count and the bf16
    combine's unit counter and warps-done count (used at this shape) are back
    at zero (the scatter's token counter is zeroed by the second barrier,
    before any CTA takes from it, so its end value does not matter), and five
    repeated steps give the same bytes as the first."""
    from combine_warp_top_fp32_b300 import workloads

    w = workloads.WORKLOADS["capacity"]
    cfg = ep.config_from_workload(w, payload=ep.EP_PAYLOAD_INT8)
    d = workloads.generate(w, device="cuda")
    buf = ep.EpBuffers.allocate(cfg)
    buf.route_dispatch(d["logits"], d["x"])
    buf.combine(d["expert_out"])
    torch.cuda.synchronize()
    first = [t.clone() for t in (buf.payload, buf.slot_row, buf.y)]
    for _ in range(5):
        buf.route_dispatch(d["logits"], d["x"])
        buf.combine(d["expert_out"])
    torch.cuda.synchronize()
    assert ep.ep_get_error(buf.ws) == ep.EP_OK
    words = buf.ws[:512].view(torch.int32).cpu().numpy()
    assert words[64 // 4] == 0 and words[68 // 4] == 0  # the combine's unit counter, warps done
    assert words[128 // 4] == 0  # the grid barrier's arrival count
    for a, b in zip(first, (buf.payload, buf.slot_row, buf.y)):
        assert torch.equal(a, b)


# ----------------------------------------------------------------------------
# device-side index checks: bad inputs become a status code, never an access
# ----------------------------------------------------------------------------
def test_bad_expert_ids_are_reported(ep):
    T, H, E, k, R = 100, 64, 8, 2, 2
    cfg = ep.make_config(T, H, E, k, R)
    buf = ep.EpBuffers.allocate(cfg)
    idx = torch.stack([torch.arange(T) % E, (torch.arange(T) + 1) % E], 1).int().cuda()
    idx[3, 1] = 8  # out of range
    idx[7, 0] = -5  # negative
    idx[9, 1] = idx[9, 0]  # repeated within a token
    buf.topk_idx.copy_(idx)
    x = torch.randn(T, H, device="cuda").to(torch.bfloat16)
    buf.dispatch(x)
    assert ep.ep_get_error(buf.ws) == ep.EP_ERR_DEVICE_INDEX
    sr = buf.slot_row.cpu().numpy().reshape(T, k)
    assert sr[3, 1] == -1 and sr[7, 0] == -1
    N = int(buf.rank_off[-1].item())
    assert np.all((sr == -1) | ((sr >= 0) & (sr < N)))
    # the status word was cleared by the read
    assert ep.ep_get_error(buf.ws) == ep.EP_OK


def test_bad_slot_rows_are_reported(ep):
    T, H, E, k, R = 16, 64, 4, 2, 2
    cfg = ep.make_config(T, H, E, k, R)
    buf = ep.EpBuffers.allocate(cfg)
    eo = torch.ones(T * k, H, dtype=torch.bfloat16, device="cuda")
    sr = torch.arange(T * k, dtype=torch.int32, device="cuda")
    sr[5] = T * k  # one past the last row
    sr[6] = -2
    w = torch.full((T, k), 0.5, device="cuda")
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    ep.ep_combine(cfg, eo, None, ep.EP_PAYLOAD_BF16, sr, w, y, buf.ws)
    assert ep.ep_get_error(buf.ws) == ep.EP_ERR_DEVICE_INDEX
    yf = y.float().cpu().numpy()
    assert np.all(yf[2] == 0.5) and np.all(yf[3] == 0.5)  # slots 5 and 6 skipped
    assert np.all(yf[0] == 1.0)


# ----------------------------------------------------------------------------
# the fused dispatch's device-wide wait: bounded, reported, recoverable
# ----------------------------------------------------------------------------
def test_fused_wait_timeout_is_reported_and_recovers(ep):
    """With the test hook on, the one grid barrier of the fused route+dispatch
    kernel waits for a CTA that does not exist and gives up after a short
    limit: the call reports EP_ERR_TIMEOUT through ep_get_error (no hang, no
    fault), and the same workspace then serves a normal call whose outputs
    match the three-call path."""
    from combine_warp_top_fp32_b300 import workloads

    w = workloads.WORKLOADS["prefill-mid"]
    cfg = ep.config_from_workload(w, payload=ep.EP_PAYLOAD_INT8)
    d = workloads.generate(w, device="cuda", expert_out=False)
    buf = ep.EpBuffers.allocate(cfg)
    ep.ep_debug_set(ep.EP_DEBUG_ROUTE_DISPATCH_FORM, ep.EP_FORM_SINGLE)
    ep.ep_debug_set(ep.EP_DEBUG_FORCE_WAIT_TIMEOUT, 1)
    try:
        buf.route_dispatch(d["logits"], d["x"])
        assert ep.ep_get_error(buf.ws) == ep.EP_ERR_TIMEOUT
    finally:
        ep.ep_debug_set(ep.EP_DEBUG_FORCE_WAIT_TIMEOUT, 0)
    ref = ep.EpBuffers.allocate(cfg)
    ref.route(d["logits"])
    ref.dispatch(d["x"])
    torch.cuda.synchronize()
    assert ep.ep_get_error(ref.ws) == ep.EP_OK
    _assert_fused_matches(ep, cfg, ref, d["logits"], d["x"])
    try:
        buf.route_dispatch(d["logits"], d["x"])  # the workspace that timed out, reused
        torch.cuda.synchronize()
        assert ep.ep_get_error(buf.ws) == ep.EP_OK
    finally:
        ep.ep_debug_set(ep.EP_DEBUG_ROUTE_DISPATCH_FORM, ep.EP_FORM_AUTO)
    N = int(ref.rank_off[-1].item())
    assert torch.equal(ref.slot_row, buf.slot_row)
    assert torch.equal(ref.payload[:N], buf.payload[:N])

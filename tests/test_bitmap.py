"""Compact routing metadata (MoE sparse-communication article,
intelliparadigm.com, §4.1: [expert, position, data] becomes [bitmap, data]).

On the host: the metadata sizes the bitmap replaces. On the GPU:
ep_bitmap_encode writes exactly the bits of the top-k ids, and
ep_bitmap_layout, from the bitmaps alone, rebuilds the oracle's layout —
counts, capacity drops, offsets — and the source token of every row
(the oracle's row_slot // k), on the workloads and edge cases."""
import numpy as np
import pytest
import torch

from combine_warp_top_fp32_b300 import workloads


def _words(E):
    return (E + 31) // 32


def metadata_bytes(E, k):
    """Per token: k (expert id, position) pairs of 4 + 4 bytes, or one bitmap."""
    return k * 8, 4 * _words(E)


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_bitmap_is_smaller_than_index_pairs(name):
    w = workloads.WORKLOADS[name]
    pairs, bitmap = metadata_bytes(w.E, w.k)
    assert bitmap < pairs  # tiny: 4 vs 16; capacity: 16 vs 64; large: 32 vs 64
    assert bitmap * 8 >= w.E


def _numpy_bitmap(idx, E):
    T, k = idx.shape
    bm = np.zeros((T, _words(E)), np.uint32)
    for j in range(k):
        e = idx[:, j].astype(np.int64)
        np.bitwise_or.at(bm, (np.arange(T), e // 32), (np.uint32(1) << (e % 32).astype(np.uint32)))
    return bm


def _ep():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from combine_warp_top_fp32_b300 import binding

    return binding


def _layout_buffers(ep, cfg):
    i32 = dict(dtype=torch.int32, device="cuda")
    rows = max(ep.ep_max_rows(cfg), 1)
    return dict(row_token=torch.full((rows,), -7, **i32), expert_counts=torch.empty(cfg.E, **i32),
                expert_raw=torch.empty(cfg.E, **i32), expert_off=torch.empty(cfg.E + 1, **i32),
                rank_off=torch.empty(cfg.R + 1, **i32), n_dropped=torch.empty(1, **i32),
                ws=torch.zeros(max(ep.ep_workspace_size(cfg), 256), dtype=torch.uint8, device="cuda"))


SHAPES = [  # T, E, k, R, cf
    (4096, 64, 6, 8, 0.0),
    (16384, 128, 8, 8, 1.25),
    (2000, 160, 5, 160, 0.0),
    (300, 1024, 32, 8, 0.5),
    (256, 8, 2, 2, 0.0),
    (1, 3, 3, 1, 0.0),
]


@pytest.mark.gpu
@pytest.mark.parametrize("T,E,k,R,cf", SHAPES)
def test_bitmap_encode_and_layout_match_oracle(orc, T, E, k, R, cf):
    ep = _ep()
    w = workloads.Workload("bm", T=T, H=16, E=E, k=k, R=R, capacity_factor=cf, payloads=(0,), seed=T + E,
                           sigma_bias=1.0)
    cfg = ep.config_from_workload(w)
    d = workloads.generate(w, device="cpu", expert_out=False)
    idx, _ = orc.route(d["logits"].numpy(), k)
    lay = orc.layout(idx, E, R, cf)
    b = _layout_buffers(ep, cfg)
    idx_d = torch.from_numpy(idx).cuda()
    bm = torch.zeros((T, _words(E)), dtype=torch.int32, device="cuda")
    ep.ep_bitmap_encode(cfg, idx_d, bm, b["ws"])
    ep.ep_bitmap_layout(cfg, bm, b["row_token"], b["expert_counts"], b["expert_raw"], b["expert_off"],
                        b["rank_off"], b["n_dropped"], b["ws"])
    torch.cuda.synchronize()
    assert ep.ep_get_error(b["ws"]) == ep.EP_OK
    np.testing.assert_array_equal(bm.cpu().numpy().view(np.uint32), _numpy_bitmap(idx, E))
    np.testing.assert_array_equal(b["expert_counts"].cpu().numpy(), lay["expert_counts"])
    np.testing.assert_array_equal(b["expert_raw"].cpu().numpy(), lay["expert_raw"])
    np.testing.assert_array_equal(b["expert_off"].cpu().numpy(), lay["expert_off"])
    np.testing.assert_array_equal(b["rank_off"].cpu().numpy(), lay["rank_off"])
    assert int(b["n_dropped"].item()) == lay["n_dropped"]
    N = lay["N"]
    np.testing.assert_array_equal(b["row_token"][:N].cpu().numpy(), lay["row_slot"] // k)


@pytest.mark.gpu
def test_bitmap_layout_of_an_empty_batch():
    ep = _ep()
    cfg = ep.make_config(0, 16, 8, 2, 2)
    b = _layout_buffers(ep, cfg)
    b["expert_off"].fill_(5)
    b["rank_off"].fill_(5)
    ep.ep_bitmap_layout(cfg, torch.empty((0, 1), dtype=torch.int32, device="cuda"), b["row_token"],
                        b["expert_counts"], b["expert_raw"], b["expert_off"], b["rank_off"], b["n_dropped"], b["ws"])
    torch.cuda.synchronize()
    assert b["expert_off"].cpu().tolist() == [0] * 9 and b["rank_off"].cpu().tolist() == [0] * 3
    assert ep.ep_get_error(b["ws"]) == ep.EP_OK


@pytest.mark.gpu
def test_bad_bitmaps_and_ids_are_reported():
    ep = _ep()
    T, E, k, R = 64, 40, 3, 2
    cfg = ep.make_config(T, 16, E, k, R)
    b = _layout_buffers(ep, cfg)
    idx = np.stack([np.arange(T) % E, (np.arange(T) + 1) % E, (np.arange(T) + 2) % E], 1).astype(np.int32)
    bm = torch.from_numpy(_numpy_bitmap(idx, E).view(np.int32)).cuda()
    ep.ep_bitmap_layout(cfg, bm, b["row_token"], b["expert_counts"], b["expert_raw"], b["expert_off"],
                        b["rank_off"], b["n_dropped"], b["ws"])
    assert ep.ep_get_error(b["ws"]) == ep.EP_OK
    for t, fix in ((5, lambda r: r & ~np.uint32(1 << 5)),  # one bit too few
                   (9, lambda r: r | np.uint32(1 << 30)),  # one too many
                   (11, lambda r: r | np.uint32(1 << 31))):  # an expert id >= E (bit 63 of 64)
        bad = _numpy_bitmap(idx, E)
        bad[t, 0 if t != 11 else 1] = fix(bad[t, 0 if t != 11 else 1])
        ep.ep_bitmap_layout(cfg, torch.from_numpy(bad.view(np.int32)).cuda(), b["row_token"], b["expert_counts"],
                            b["expert_raw"], b["expert_off"], b["rank_off"], b["n_dropped"], b["ws"])
        assert ep.ep_get_error(b["ws"]) == ep.EP_ERR_DEVICE_INDEX, t
    idx_bad = idx.copy()
    idx_bad[3, 1] = E + 4
    ep.ep_bitmap_encode(cfg, torch.from_numpy(idx_bad).cuda(), torch.empty((T, 2), dtype=torch.int32, device="cuda"),
                        b["ws"])
    assert ep.ep_get_error(b["ws"]) == ep.EP_ERR_DEVICE_INDEX

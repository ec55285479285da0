"""MoE expert path on the GPU against the oracle, stage by stage.

(a)+(b) dispatch: global scale, routing arrays and the permuted quantised rows
        bit-exact;
(c)     w13 GEMM + SiLU*up: fp32 h (debug dump) within the GEMM bound on
        identical operands; re-quantised codes agree with the oracle's except
        at rounding ties (rate reported, >= 99.9 %);
(d)     w2 GEMM + weighted scatter-add run on the oracle's own re-quantised h
        (written into the workspace), so its output is on identical operands;
full    nvfp4_moe_forward: tokens whose re-quantised rows all match the
        oracle's are held to the GEMM bound, the whole output to cosine 0.999.
Tiny configurations are checked on every token; the 384-expert decode and
prefill workloads (the prefill ones with the benchmark's seeds) on sampled
tokens.
"""

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_quant_gb300 import _lib, model, ops, workloads
from oracle import nvfp4_oracle as O
from tests.helpers import assert_parity, bf16_to_np, oracle_expert_fn, oracle_pool

pytestmark = pytest.mark.gpu
DEV = "cuda"
F32 = np.float32


def _region(ws, off, n, dtype):
    nbytes = n * torch.empty(0, dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype)


def calibrate_a2(res: O.MoEResult, E: int) -> np.ndarray:
    """Static scale of the intermediate: fl32(max |h| / 2688) over the rows the oracle computed."""
    amax = max(float(np.max(np.abs(r.h))) for r in res.rows.values())
    return np.full(E + 1, F32(F32(amax) / F32(2688.0)), dtype=np.float32)


def run_moe_check(x, ids, w, W: ops.MoEWeights, oe, tokens, shared: bool, strict_all=False, mapper=map,
                  calib_tokens=None):
    """Stage-by-stage check of the tokens listed.  The static scale of h is calibrated on
    ``calib_tokens`` (default: the tokens checked); rows of other tokens whose h exceeds it
    saturate their E4M3 scale identically on both sides.  ``mapper`` runs the oracle's
    per-expert jobs (a process pool's imap for the full-size workloads)."""
    T, H = x.shape
    k = ids.shape[1]
    E, I = W.E, W.I
    xnp, idsnp, wnp = x.float().numpy(), ids.numpy(), w.numpy()
    sh = oe(E) if shared else None
    cal = O.moe_forward(xnp, idsnp, wnp, oe, E, np.ones(E + 1, F32), shared=sh,
                        tokens=tokens if calib_tokens is None else calib_tokens, mapper=mapper)
    a2 = calibrate_a2(cal, E)
    ref = O.moe_forward(xnp, idsnp, wnp, oe, E, a2, shared=sh, tokens=tokens, mapper=mapper)

    xd, idsd, wd, a2d = x.to(DEV), ids.to(DEV), w.to(DEV), torch.from_numpy(a2).to(DEV)
    L = ops.moe_workspace_layout(T, H, I, E, k, shared)
    ws = torch.empty(L.total, dtype=torch.uint8, device=DEV)
    a1 = torch.empty(1, dtype=torch.float32, device=DEV)

    # ---------------------------------------------------------------- (a) + (b)
    ops.moe_dispatch(xd, idsd, W, a1, True, ws)
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    assert a1.item() == float(ref.xq.gs), "a1 global scale"
    G = E + int(shared)
    counts = _region(ws, L.counts, G, torch.int32).cpu().numpy()
    offsets = _region(ws, L.offsets, G + 1, torch.int32).cpu().numpy()
    pad = _region(ws, L.pad_offsets, G + 1, torch.int32).cpu().numpy()
    tiles = _region(ws, L.tile_offsets, G + 1, torch.int32).cpu().numpy()
    sorted_idx = _region(ws, L.sorted_idx, T * k, torch.int32).cpu().numpy()
    inv_idx = _region(ws, L.inv_idx, T * k, torch.int32).cpu().numpy()
    want_counts = np.concatenate([ref.routing.counts, [T] if shared else []]).astype(np.int64)
    np.testing.assert_array_equal(counts, want_counts)
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(want_counts)]))
    np.testing.assert_array_equal(pad, np.concatenate([[0], np.cumsum((want_counts + 127) // 128 * 128)]))
    R = 32 if T <= 128 else 128  # m-tile height: 32-row tiles up to 128 tokens
    np.testing.assert_array_equal(tiles, np.concatenate([[0], np.cumsum((want_counts + R - 1) // R)]))
    # the GEMMs' schedule: per tile (group, tile in group | bit 30 when the group spans several
    # tiles, live rows, first permuted row)
    table = _region(ws, L.tile_table, 4 * int(tiles[-1]), torch.int32).view(-1, 4).cpu().numpy()
    want_table = [(g, mt | ((1 << 30) if c > R else 0), min(R, c - mt * R), int(pad[g]) + mt * R)
                  for g, c in enumerate(want_counts.tolist()) for mt in range((c + R - 1) // R)]
    np.testing.assert_array_equal(table, np.array(want_table, dtype=np.int64).reshape(-1, 4))
    np.testing.assert_array_equal(sorted_idx, ref.routing.sorted_idx)
    np.testing.assert_array_equal(inv_idx, ref.routing.inv_idx)
    dest_rows = _region(ws, L.dest_rows, T * k, torch.int32).cpu().numpy()
    flat_e = idsnp.reshape(-1)
    np.testing.assert_array_equal(dest_rows, pad[flat_e] + ref.routing.inv_idx - offsets[flat_e])

    rc = L.rows_capacity
    xq = _region(ws, L.xq, rc * H // 2, torch.uint8).view(rc, H // 2)
    xsf = _region(ws, L.xsf, O.sf_bytes(rc, H), torch.uint8).cpu().numpy()
    xsf_off = O.sf_swizzle_offsets(rc, H)

    def row_of(t, j):
        if j < 0:
            return int(pad[E]) + t
        f = t * k + j
        e = int(ids[t, j])
        return int(pad[e]) + int(inv_idx[f]) - int(offsets[e])

    slots = [(t, j) for t in tokens for j in list(range(k)) + ([-1] if shared else [])]
    rows = np.array([row_of(t, j) for t, j in slots])
    xq_rows = O.unpack_codes(xq[torch.from_numpy(rows).to(DEV)].cpu().numpy())
    tok = np.array([t for t, _ in slots])
    np.testing.assert_array_equal(xq_rows, ref.xq.codes[tok])
    np.testing.assert_array_equal(xsf[xsf_off[rows, : H // 16]], ref.xq.sf[tok])

    # ---------------------------------------------------------------- (c)
    h_dbg = torch.full((rc, I), float("nan"), dtype=torch.float32, device=DEV)
    ops.moe_w13(T, k, W, a1, a2d, ws, h_debug=h_dbg)
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    h_gpu = h_dbg[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    h_ref = np.stack([ref.rows[s].h[0] for s in slots])
    assert_parity(h_gpu, h_ref, what="w13 SiLU(gate)*up")
    hq = _region(ws, L.hq, rc * I // 2, torch.uint8).view(rc, I // 2)
    hsf_t = _region(ws, L.hsf, O.sf_bytes(rc, I), torch.uint8)
    hsf = hsf_t.cpu().numpy()
    hsf_off = O.sf_swizzle_offsets(rc, I)
    hq_gpu = O.unpack_codes(hq[torch.from_numpy(rows).to(DEV)].cpu().numpy())
    hq_ref = np.stack([ref.rows[s].hq.codes[0] for s in slots])
    hsf_gpu = hsf[hsf_off[rows, : I // 16]]
    hsf_ref = np.stack([ref.rows[s].hq.sf[0] for s in slots])
    code_agree = float(np.mean(hq_gpu == hq_ref))
    sf_agree = float(np.mean(hsf_gpu == hsf_ref))
    assert code_agree >= 0.999 and sf_agree >= 0.999, (code_agree, sf_agree)
    row_match = np.all(hq_gpu == hq_ref, axis=1) & np.all(hsf_gpu == hsf_ref, axis=1)

    hq_split = hq[torch.from_numpy(rows).to(DEV)].cpu().numpy()  # the stage-by-stage w13's rows
    hsf_split = hsf_gpu.copy()

    # ---------------------------------------------------------------- (d) on the oracle's operands
    hq_host = hq.cpu().numpy()
    hq_host[rows] = O.pack_codes(hq_ref)
    hq.copy_(torch.from_numpy(hq_host).to(DEV))
    hsf[hsf_off[rows, : I // 16]] = hsf_ref
    hsf_t.copy_(torch.from_numpy(hsf).to(DEV))
    ops.moe_w2(T, k, wd, W, a2d, ws)
    y_stage = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    ops.moe_finalize(T, k, W, y_stage, ws)
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    assert_parity(bf16_to_np(y_stage)[tokens], ref.y, what="w2 + scatter-add on identical operands")

    # ---------------------------------------------------------------- full forward
    y, g = ops.moe_forward(xd, idsd, wd, W, a2d, workspace=ws)
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    assert g.item() == float(ref.xq.gs)
    # the forward's w13 (at T = 1 the one-token kernel, which quantises x itself and takes its
    # schedule from the ids) leaves the same re-quantised rows as the stage-by-stage launches
    np.testing.assert_array_equal(hq[torch.from_numpy(rows).to(DEV)].cpu().numpy(), hq_split)
    np.testing.assert_array_equal(hsf_t.cpu().numpy()[hsf_off[rows, : I // 16]], hsf_split)
    yf = bf16_to_np(y)[tokens]
    assert np.isfinite(bf16_to_np(y)).all()
    slot_tok = np.array([tokens.index(t) for t, _ in slots])
    clean = np.array([row_match[slot_tok == i].all() for i in range(len(tokens))])
    if clean.any():
        assert_parity(yf[clean], ref.y[clean], what="forward, tokens with identical re-quantised rows")
    if strict_all:
        assert clean.all(), f"{(~clean).sum()} tokens with a re-quantisation tie"
    assert O.cosine(yf, ref.y) >= 0.999
    return dict(code_agree=code_agree, sf_agree=sf_agree, clean_tokens=int(clean.sum()), tokens=len(tokens))


@pytest.mark.parametrize("cfg", [workloads.TINY, workloads.TINY_SHARED])
def test_moe_tiny_all_tokens(cfg):
    base = 101
    W = model.make_moe_weights(cfg.E, cfg.H, cfg.I, base, DEV, shared=cfg.shared)
    oe = oracle_expert_fn(base, cfg.H, cfg.I, DEV)
    x = workloads.activations(cfg.T, cfg.H, seed=102, device="cpu")
    ids, w = workloads.routing(cfg, seed=103, device="cpu")
    run_moe_check(x, ids, w, W, oe, list(range(cfg.T)), cfg.shared)


def test_moe_tiny_duplicates_and_skew():
    """All tokens on one expert (a 128+ row segment spans two m tiles) and duplicate ids in a token."""
    T, H, I, E, k = 150, 256, 128, 4, 2
    base = 104
    W = model.make_moe_weights(E, H, I, base, DEV, shared=True)
    oe = oracle_expert_fn(base, H, I, DEV)
    x = workloads.activations(T, H, seed=105, device="cpu")
    ids = torch.zeros(T, k, dtype=torch.int32)
    ids[::3, 1] = 2
    ids[1::3, 0] = 3
    ids[1::3, 1] = 3  # duplicate expert within a token
    w = torch.softmax(torch.randn(T, k, generator=torch.Generator().manual_seed(1)), -1).contiguous()
    run_moe_check(x, ids, w, W, oe, list(range(0, T, 7)), True)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 33, 128, 129])
def test_moe_small_batches_all_tokens(T):
    """Small calls, all tokens: up to 128 tokens the groups are cut into 32-row tiles and the
    GEMMs take the ring with 4 small A stages (one 32-row box per tile); at T = 128 the 16
    experts hold about 64 rows each and the shared one 128, so their tiles start 32, 64 and
    96 rows into a scale block.  T = 129 takes 128-row tiles and the regular ring."""
    cfg = workloads.MoEConfig("small", T, 256, 128, 16, 8, True, "softmax", False)
    base = 109
    W = model.make_moe_weights(cfg.E, cfg.H, cfg.I, base, DEV, shared=True)
    oe = oracle_expert_fn(base, cfg.H, cfg.I, DEV)
    x = workloads.activations(T, cfg.H, seed=110 + T, device="cpu")
    ids, w = workloads.routing(cfg, seed=120 + T, device="cpu")
    run_moe_check(x, ids, w, W, oe, list(range(T)), True)


@pytest.mark.parametrize("T,E,k,mode", [(32, 4, 8, "random"), (20, 2, 8, "random"), (32, 1, 8, "same"),
                                         (9, 2, 8, "random")])
def test_moe_small_batch_duplicate_ids(T, E, k, mode):
    """Up to 32 tokens, with ids repeated inside a token: a group then holds more than T rows and
    spans several 32-row tiles, which start 32, 64 or 96 rows into a 128-row scale block (the
    A scales are rotated into place) and run past the first block.  All tokens are checked."""
    H, I = 256, 128
    base = 131
    W = model.make_moe_weights(E, H, I, base, DEV, shared=True)
    oe = oracle_expert_fn(base, H, I, DEV)
    x = workloads.activations(T, H, seed=132 + T, device="cpu")
    rng = np.random.default_rng(133 + T * E)
    if mode == "same":
        ids = torch.zeros(T, k, dtype=torch.int32)
    else:
        ids = torch.from_numpy(rng.integers(0, E, (T, k)).astype(np.int32))
    w = torch.softmax(torch.from_numpy(rng.standard_normal((T, k)).astype(np.float32)), -1).contiguous()
    counts = np.bincount(ids.numpy().reshape(-1), minlength=E)
    assert counts.max() > 32, "the case must put more than 32 rows in a group"
    run_moe_check(x, ids, w, W, oe, list(range(T)), True)


@pytest.mark.parametrize("T", [2, 9])
def test_moe_dispatch_static_gs(T):
    """Static a1 scale: every routed and shared row holds the oracle's codes."""
    H, I, E, k = 256, 128, 8, 2
    W = model.make_moe_weights(E, H, I, 111, DEV, shared=True)
    x = workloads.activations(T, H, seed=112, device="cpu")
    ids = torch.from_numpy(np.random.default_rng(T).integers(0, E, (T, k)).astype(np.int32))
    L = ops.moe_workspace_layout(T, H, I, E, k, True)
    ws = torch.empty(L.total, dtype=torch.uint8, device=DEV)
    gs = 0.003
    ops.moe_dispatch(x.to(DEV), ids.to(DEV), W, torch.tensor([gs], dtype=torch.float32, device=DEV), False, ws)
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    ref = O.quantize(x.float().numpy(), gs=F32(gs))
    rc = L.rows_capacity
    xq = O.unpack_codes(_region(ws, L.xq, rc * H // 2, torch.uint8).view(rc, H // 2).cpu().numpy())
    xsf = _region(ws, L.xsf, O.sf_bytes(rc, H), torch.uint8).cpu().numpy()
    off = O.sf_swizzle_offsets(rc, H)
    dest = _region(ws, L.dest_rows, T * k, torch.int32).cpu().numpy().reshape(T, k)
    pad = _region(ws, L.pad_offsets, E + 2, torch.int32).cpu().numpy()
    for t in range(T):
        for p in list(dest[t]) + [pad[E] + t]:
            np.testing.assert_array_equal(xq[p], ref.codes[t])
            np.testing.assert_array_equal(xsf[off[p, : H // 16]], ref.sf[t])


def test_moe_empty_batch():
    W = model.make_moe_weights(4, 256, 128, 106, DEV, shared=True)
    y, g = ops.moe_forward(torch.empty(0, 256, dtype=torch.bfloat16, device=DEV),
                           torch.empty(0, 2, dtype=torch.int32, device=DEV),
                           torch.empty(0, 2, dtype=torch.float32, device=DEV), W,
                           torch.full((5,), 0.01, device=DEV))
    torch.cuda.synchronize()
    assert y.shape == (0, 256) and g.item() == 0.0


@pytest.fixture(scope="module")
def big_weights():
    cfg = workloads.PREFILL
    W = model.make_moe_weights(cfg.E, cfg.H, cfg.I, workloads.BENCH_WEIGHT_SEED, DEV, shared=True)
    oe = oracle_expert_fn(workloads.BENCH_WEIGHT_SEED, cfg.H, cfg.I, DEV)
    yield W, oe
    del W
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def oracle_map():
    """The oracle's per-expert jobs of the full-size workloads run in a spawned process pool."""
    pool = oracle_pool()

    def mapper(fn, jobs):
        it = pool.imap(fn, jobs, chunksize=1)
        for _ in range(len(jobs)):
            yield it.next(timeout=900)  # a worker that cannot start fails the test, not hangs it

    yield mapper
    pool.terminate()
    pool.join()


def segment_rows(ids: np.ndarray, e: int) -> np.ndarray:
    """Tokens of expert e's routed rows in segment order (the routing is stable by flat index)."""
    k = ids.shape[1]
    return np.nonzero(ids.reshape(-1) == e)[0] // k


@pytest.mark.parametrize("ids_row,shared", [([3, 3, 1, 3, 0, 1, 2, 3], True), ([5, 2, 7, 5, 0, 6, 1, 4], False),
                                            ([6, 6, 6, 6, 6, 6, 6, 6], True)])
def test_moe_one_token_repeated_ids(ids_row, shared):
    """One token (the one-token w13: x quantised in the GEMM CTAs, schedule from the ids) with an
    expert listed up to eight times: that group's tile holds as many copies of the token."""
    H, I, E, k = 384, 128, 8, 8  # H = 384: the last K stage holds two of its four K steps
    base = 141
    W = model.make_moe_weights(E, H, I, base, DEV, shared=shared)
    oe = oracle_expert_fn(base, H, I, DEV)
    x = workloads.activations(1, H, seed=142, device="cpu", outliers=True)
    ids = torch.tensor([ids_row], dtype=torch.int32)
    w = torch.softmax(torch.randn(1, k, generator=torch.Generator().manual_seed(143)), -1).contiguous()
    run_moe_check(x, ids, w, W, oe, [0], shared)


def test_moe_one_token_dirty_workspace():
    """One token on a workspace full of stale bytes: the routing zeroes the fp32 accumulator
    that the one-token launch adds into, so two calls in a row on the same workspace give the
    zeroed workspace's y."""
    H, I, E, k = 512, 128, 8, 4
    W = model.make_moe_weights(E, H, I, 161, DEV, shared=True)
    x = workloads.activations(1, H, seed=162, device=DEV)
    ids = torch.tensor([[2, 7, 0, 5]], dtype=torch.int32, device=DEV)
    w = torch.softmax(torch.randn(1, k, generator=torch.Generator().manual_seed(163)), -1).to(DEV)
    a2 = torch.full((E + 1,), 0.01, device=DEV)
    L = ops.moe_workspace_layout(1, H, I, E, k, True)
    y0, _ = ops.moe_forward(x, ids, w, W, a2, workspace=torch.zeros(L.total, dtype=torch.uint8, device=DEV))
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    assert float(y0.float().abs().max()) > 0
    ws = torch.full((L.total,), 0xFF, dtype=torch.uint8, device=DEV)
    y = torch.empty(1, H, dtype=torch.bfloat16, device=DEV)
    for _ in range(2):
        y.fill_(float("nan"))
        ops.moe_forward(x, ids, w, W, a2, workspace=ws, out=y)
        torch.cuda.synchronize()
        assert ops.device_error() == (0, 0)
        assert bool(torch.isfinite(y.float()).all())
        np.testing.assert_allclose(bf16_to_np(y), bf16_to_np(y0), rtol=1e-2, atol=1e-3 * float(y0.float().abs().max()))


def test_moe_one_token_static_gs_and_bad_id():
    """One token: a static a1 scale equal to the dynamic one gives the same re-quantised rows; an
    out-of-range id is dropped (the routing flags it) and the w13 schedule drops it too."""
    H, I, E, k = 512, 128, 8, 4
    W = model.make_moe_weights(E, H, I, 151, DEV, shared=True)
    x = workloads.activations(1, H, seed=152, device=DEV)
    ids = torch.tensor([[4, 1, 6, 2]], dtype=torch.int32, device=DEV)
    w = torch.full((1, k), 0.25, device=DEV)
    a2 = torch.full((E + 1,), 0.01, device=DEV)
    L = ops.moe_workspace_layout(1, H, I, E, k, True)
    ws = torch.zeros(L.total, dtype=torch.uint8, device=DEV)
    hq = _region(ws, L.hq, L.rows_capacity * I // 2, torch.uint8)
    y_dyn, g = ops.moe_forward(x, ids, w, W, a2, workspace=ws)
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    hq_dyn = hq.clone()
    hq.zero_()
    y_st, _ = ops.moe_forward(x, ids, w, W, a2, a1_gs=g.clone(), workspace=ws)
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    assert torch.equal(hq, hq_dyn)
    assert torch.allclose(y_st.float(), y_dyn.float(), rtol=1e-2, atol=1e-3)
    ids_bad = ids.clone()
    ids_bad[0, 2] = 9
    ops.device_error()
    y_bad, _ = ops.moe_forward(x, ids_bad, w, W, a2, workspace=ws)
    st, flags = ops.device_error()
    assert st == _lib.ERR_DEVICE_FAULT and flags == _lib.DEVERR_BAD_EXPERT_ID
    w_drop = w.clone()
    w_drop[0, 2] = 0.0
    y_drop, _ = ops.moe_forward(x, ids, w_drop, W, a2, workspace=ws)
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    assert torch.allclose(y_bad.float(), y_drop.float(), rtol=1e-2, atol=1e-3)


def chunk_tokens(ids: np.ndarray, n: int, seed: int, R: int = 32) -> list:
    """At least n tokens of a 128-token chunk that reach every kind of m tile: one token in each
    R-row tile of the shared expert (its row i is token i), the last row of every tile of the two
    most popular experts (groups of several tiles, later ones with rotated A scales), a token of a
    one-row group; seeded others fill up to n."""
    T = ids.shape[0]
    counts = np.bincount(ids.reshape(-1), minlength=int(ids.max()) + 1)
    chosen = {tile * R + (7 * tile + 3) % R for tile in range(T // R)}
    hot = np.argsort(-counts, kind="stable")[:2]
    assert counts[hot[0]] > R, "the chunk must hold a group of several tiles"
    for e in hot:
        toks = segment_rows(ids, int(e))
        chosen.update(int(toks[min(len(toks) - 1, t * R + R - 1)]) for t in range((len(toks) + R - 1) // R))
    single = np.nonzero(counts == 1)[0]
    assert len(single), "the chunk must hold a one-row group"
    chosen.add(int(segment_rows(ids, int(single[0]))[0]))
    rng = np.random.default_rng(seed)
    while len(chosen) < n:
        chosen.add(int(rng.integers(0, T)))
    return sorted(chosen)


@pytest.mark.parametrize("T", [1, 8, 64])
def test_moe_decode_all_tokens(big_weights, oracle_map, T):
    """The decode batches of the 384-expert layer (32-row tiles, the small-A ring), every token."""
    W, oe = big_weights
    x, ids, w = workloads.decode_step(T, device="cpu")
    run_moe_check(x, ids, w, W, oe, list(range(T)), True, mapper=oracle_map, calib_tokens=[0])


@pytest.mark.parametrize("chunk", [0, 31])
def test_moe_prefill_bench_chunk_tiles(big_weights, oracle_map, chunk):
    """Prefill chunks of the benchmark (its seeds and weights): 16+ tokens covering every 32-row
    tile of the shared expert, every tile of the two most popular experts and a one-row group."""
    W, oe = big_weights
    x, ids, w = workloads.prefill_chunk(chunk, device="cpu")
    tokens = chunk_tokens(ids.numpy(), 16, seed=chunk)
    assert len(tokens) >= 16
    run_moe_check(x, ids, w, W, oe, tokens, True, mapper=oracle_map, calib_tokens=tokens[:2])


def test_moe_prefill_whole_4096_hot_experts(big_weights, oracle_map):
    """4096 tokens in one call (128-row tiles; the hottest experts span many m tiles and re-read
    their weights from L2): the last row of each of the three hottest experts, the first and last
    token and seeded others."""
    W, oe = big_weights
    x, ids, w = workloads.prefill_whole(device="cpu")
    idn = ids.numpy()
    counts = np.bincount(idn.ravel(), minlength=384)
    assert counts.max() > 1000  # the hottest expert spans 8+ m tiles
    hot = np.argsort(-counts, kind="stable")[:3]
    tokens = {0, x.shape[0] - 1} | {int(segment_rows(idn, int(e))[-1]) for e in hot}
    rng = np.random.default_rng(4096)
    while len(tokens) < 8:
        tokens.add(int(rng.integers(0, x.shape[0])))
    tokens = sorted(tokens)
    run_moe_check(x, ids, w, W, oe, tokens, True, mapper=oracle_map, calib_tokens=tokens[:2])


@pytest.mark.parametrize("T", [16, 1])
def test_moe_forward_cuda_graph_replay(T):
    """nvfp4_moe_forward captured in a CUDA graph and replayed matches eager execution; new inputs
    and routings written into the captured buffers flow through the replay (T = 1: the one-token
    launch, which reads the ids before its dependency wait)."""
    base = workloads.TINY_SHARED
    cfg = workloads.MoEConfig(base.name, T, base.H, base.I, base.E, base.topk, True, base.routing, False)
    W = model.make_moe_weights(cfg.E, cfg.H, cfg.I, 108, DEV, shared=True)
    ws = ops.moe_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk, True, DEV)
    a2 = torch.full((cfg.E + 1,), 0.004, device=DEV)
    x = workloads.activations(cfg.T, cfg.H, seed=1, device=DEV)
    ids, w = workloads.routing(cfg, seed=2, device=DEV)
    y = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=DEV)
    gs = torch.empty(1, device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):  # warm-up outside the capture (per-device set-up, kernel attributes)
            ops.moe_forward(x, ids, w, W, a2, workspace=ws, out=y)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = y.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ops.moe_forward(x, ids, w, W, a2, workspace=ws, out=y)
    y.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert ops.device_error() == (0, 0)
    # replays differ from eager only in the fp32 atomic summation order
    np.testing.assert_allclose(bf16_to_np(y), bf16_to_np(eager), rtol=1e-2, atol=1e-3 * float(eager.float().abs().max()))
    # new inputs in the captured buffers flow through the replay
    x.copy_(workloads.activations(cfg.T, cfg.H, seed=3, device=DEV))
    ids2, w2 = workloads.routing(cfg, seed=4, device=DEV)
    ids.copy_(ids2)
    w.copy_(w2)
    g.replay()
    y2 = y.clone()
    ops.moe_forward(x, ids, w, W, a2, workspace=ws, out=y)
    torch.cuda.synchronize()
    np.testing.assert_allclose(bf16_to_np(y2), bf16_to_np(y), rtol=1e-2, atol=1e-3 * float(y.float().abs().max()))

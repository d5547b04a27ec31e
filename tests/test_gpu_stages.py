"""GPU parity, stage by stage, on small seeded cases that span several tiles and ragged tails.

Each stage of the CUDA path is compared with the oracle on byte-identical inputs: the oracle's
indexer reads the GPU's compressed key pool, its top-k reads the GPU's scores, its attention reads
the GPU's pools and top-k indices.  Tolerances are the ones stated in tests/_parity.py.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_c4a_gb300 import dsa, synth
from compressed_sparse_attention_c4a_gb300.step import LayerStep, SM_SCALE
from oracle import layer as OL, attention as OA
from _parity import (ATTN_REL_L2, assert_attn_close, attn_bound, pool_absmax, ROW_REL_L2, np64, rel_l2, to_device, oracle_pool, idx_pool,
                     rolling_states,
                     new_tokens, pool_rows, topk_sets_match, check_rows, check_pool_rows)

pytestmark = pytest.mark.gpu
S = synth.CaseSpec

CASES = {
    # decode, ragged contexts: one below k visible entries, one at a 256-position block boundary
    "c4a_decode": S("c4a_decode", cached=[1000, 2999, 777, 4095], new=[1] * 4, seed=11),
    # bulk compression from an empty cache (the tiny-layer shape at reduced length)
    "c4a_bulk": S("c4a_bulk", cached=[0], new=[700], heads=16, idx_heads=4, idx_dim=64, index_compress=False,
                  seed=12),
    # chunked prefill whose first entry straddles the cached tokens (state ring) and the chunk
    "c4a_chunk": S("c4a_chunk", cached=[1037], new=[300], queries="all", seed=13),
    "c4a_multi_prefill": S("c4a_multi_prefill", cached=[300, 515], new=[64, 32], queries="all", heads=32, seed=14),
    # c128a: dense over entries; context 128 sees exactly its first entry
    "c128a_decode": S("c128a_decode", kind="c128a", cached=[5000, 1279, 127], new=[1] * 3, idx_heads=0, topk=0,
                      seed=15),
    "c128a_fp8": S("c128a_fp8", kind="c128a", cached=[3000, 640], new=[1] * 2, idx_heads=0, topk=0,
                   main_dtype="fp8", swa_dtype="fp8", seed=16),
    "c128a_chunk": S("c128a_chunk", kind="c128a", cached=[300], new=[200], queries="all", idx_heads=0, topk=0,
                     seed=17),
    # the method's first positions ([P2] 机制四): queries m = 0 .. 299 of a fresh request, so m < 7 sees no c4a
    # entry (an empty score row, a top-k row of -1) and m < 127 a window shorter than 128 tokens
    "c4a_early": S("c4a_early", cached=[0], new=[300], queries="all", seed=20),
    # c128a from position 0: no entry before m = 127, the first one at m = 127, the second at m = 255
    "c128a_early": S("c128a_early", kind="c128a", cached=[0], new=[300], queries="all", idx_heads=0, topk=0,
                     seed=21),
    # fp4 (e2m1) indexer keys ([P2] 第三层): the compressor writes packed codes, the indexer's tensor cores read them
    "c4a_decode_fp4": S("c4a_decode_fp4", cached=[1000, 2999, 777, 4095, 130], new=[1] * 5, idx_dtype="fp4",
                        seed=22),
    "c4a_chunk_fp4": S("c4a_chunk_fp4", cached=[1037, 64], new=[300, 75], queries="all", idx_dtype="fp4", seed=23),
    # per-channel compressor gate (one logit per raw token and channel), decode, chunk (ring + chunk) and c128a
    "c4a_decode_pc": S("c4a_decode_pc", cached=[1000, 2999, 777, 6], new=[1] * 4, gate="channel", seed=24),
    "c4a_chunk_pc": S("c4a_chunk_pc", cached=[1037, 3], new=[300, 40], queries="all", gate="channel", seed=25),
    "c128a_chunk_pc": S("c128a_chunk_pc", kind="c128a", cached=[300, 64], new=[200, 130], queries="all", idx_heads=0,
                        topk=0, gate="channel", seed=26),
}
INDEXED = [n for n, s in CASES.items() if s.idx_heads]


def _setup(name):
    cpu = synth.make_case(CASES[name], "cpu")
    gpu = to_device(cpu)
    return cpu, gpu, LayerStep(gpu)


def _oracle_compress(cpu, which, record=None):
    spec = cpu["spec"]
    epb = cpu["epb"]
    if which == "main":
        pool = oracle_pool(cpu["main_data"], cpu["main_scale"], epb)
        swa = oracle_pool(cpu["swa_data"], cpu["swa_scale"], 256)
        bt, swa_bt = np64(cpu["bt_main"]), np64(cpu["bt_swa"])
        rope_dim = spec.rope_dim
    else:
        pool = idx_pool(cpu)
        swa, bt, swa_bt = None, np64(cpu["bt_idx"]), None
        rope_dim = min(spec.rope_dim, spec.idx_dim)
    states = rolling_states(cpu, which)
    xs, zs = new_tokens(cpu, which)
    emitted = OL.compress(spec.kind, np64(cpu["start_pos"]), xs, zs, states, rope_dim, pool, bt, swa, swa_bt,
                          record=record)
    return pool, swa, states, emitted


@pytest.mark.parametrize("name", list(CASES))
def test_compress_main_and_swa(name):
    """Every emitted entry and every new token's window row, row by row; the rolling state bit for bit."""
    cpu, gpu, step = _setup(name)
    step.compress()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    rec = {}
    pool, swa, states, emitted = _oracle_compress(cpu, "main", rec)
    spec, epb = cpu["spec"], cpu["epb"]
    bt = np64(cpu["bt_main"])
    prows, vals, stored = [], [], []
    for r, ids in enumerate(emitted):
        for i in ids:
            prows.append(int(bt[r][i // epb]) * epb + i % epb)
            vals.append(rec[("entry", r, i)])
            stored.append(pool.read(bt[r], [i])[0])
    if prows:
        check_pool_rows(gpu["main_data"], gpu["main_scale"], prows, vals, stored)
    # the first entry a chunk closes spans tokens of the rolling state and of the chunk (when there is one)
    start = np64(cpu["start_pos"])
    w, st_ = synth.WINDOW[spec.kind]
    for r, ids in enumerate(emitted):
        if ids and start[r] > 0 and st_ * ids[0] < start[r]:
            assert st_ * ids[0] + w - 1 >= start[r]          # the straddling entry was among those checked
    # SWA rows of every new token
    sbt = np64(cpu["bt_swa"])
    cu = np64(cpu["cu_new"])
    prows, vals, stored = [], [], []
    for r in range(spec.batch):
        for j in range(cu[r + 1] - cu[r]):
            p = int(start[r]) + j
            prows.append(int(sbt[r][p // 256]) * 256 + p % 256)
            vals.append(rec[("swa", r, p)])
            stored.append(swa.read(sbt[r], [p])[0])
    check_pool_rows(gpu["swa_data"], gpu["swa_scale"], prows, vals, stored)
    # rolling state: a bit-exact copy of the last w raw tokens
    gx, gz = np64(gpu["state_x"]), np64(gpu["state_z"])
    for r in range(spec.batch):
        slot = int(np64(cpu["state_slot"])[r])
        assert np.array_equal(gx[slot], states[r].x) and np.array_equal(gz[slot], states[r].z)


@pytest.mark.parametrize("name", [n for n in INDEXED if CASES[n].index_compress])
def test_compress_indexer(name):
    """Indexer entries (e4m3 + amax/448 scale, or e2m1 + amax/6) code by code, row by row."""
    cpu, gpu, step = _setup(name)
    step.compress()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    rec = {}
    pool, _, states, emitted = _oracle_compress(cpu, "index", rec)
    bt = np64(cpu["bt_idx"])
    prows, vals, stored = [], [], []
    for r, ids in enumerate(emitted):
        for i in ids:
            prows.append(int(bt[r][i // 64]) * 64 + i % 64)
            vals.append(rec[("entry", r, i)])
            stored.append(pool.read(bt[r], [i])[0])
    assert prows
    check_pool_rows(gpu["idx_data"], gpu["idx_scale"], prows, vals, stored, fmt=cpu["spec"].idx_dtype)
    gx = np64(gpu["state_xi"])
    for r in range(cpu["spec"].batch):
        assert np.array_equal(gx[int(np64(cpu["state_slot"])[r])], states[r].x)


@pytest.mark.parametrize("name", ["c4a_decode", "c4a_chunk", "c4a_early", "c4a_decode_fp4", "c4a_multi_prefill",
                                  "c4a_chunk_pc"])
def test_compress_jobs_equal_separate_calls(name):
    """dsa_compress_jobs (main cache + window insert and the indexer cache in one launch) writes the same bytes
    to every pool, window row and rolling state as one dsa_compress call per cache."""
    cpu = synth.make_case(CASES[name], "cpu")
    outs = []
    for fused in (True, False):
        gpu = to_device(cpu)
        step = LayerStep(gpu)
        if fused:
            step.compress()
        else:
            step.compress_main()
            step.compress_index()
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0
        outs.append({k: gpu[k].cpu() for k in ("main_data", "swa_data", "idx_data", "idx_scale", "state_x", "state_z",
                                               "state_xi", "state_zi")})
    for k in outs[0]:
        assert torch.equal(outs[0][k], outs[1][k]), k


@pytest.mark.parametrize("name", ["c4a_decode", "c4a_multi_prefill", "c128a_early"])
def test_query_job_matches_oracle(name):
    """The query job of the compressor launch ([P2] 融合点 3): every (query, head) row is the oracle's
    query_prep (RMSNorm, then R_m) within bf16 rounding, in place or not; the compressor's outputs are those of
    the launch without it, bit for bit; and the queries alone (no compressor work) are accepted."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    cpu = synth.make_case(CASES[name], "cpu")
    spec = cpu["spec"]
    g = torch.Generator().manual_seed(99)
    q_raw = (torch.randn(cpu["q"].shape, generator=g) * 3.0).to(torch.bfloat16)
    want = OA.query_prep(np64(q_raw), np64(cpu["q_pos"])[:, None], spec.rope_dim)
    outs = []
    for mode in ("without", "with", "in_place"):
        gpu = to_device(cpu)
        step = LayerStep(gpu)
        jobs = step._jobs()
        qr = q_raw.cuda()
        qo = qr if mode == "in_place" else torch.empty_like(qr)
        qj = dsa.query_job(qr, qo, gpu["q_pos"], step.rope_main) if mode != "without" else None
        dsa.dsa_compress_jobs(step.kind, gpu["cu_new"], gpu["start_pos"], step.max_new, gpu["state_slot"],
                              gpu["state_x"].shape[0], jobs, dev_status=step.status, query=qj)
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0
        outs.append(({k: gpu[k].cpu() for k in ("main_data", "swa_data", "state_x", "state_z")}, qo.cpu()))
    for k in outs[0][0]:
        assert torch.equal(outs[0][0][k], outs[1][0][k]) and torch.equal(outs[0][0][k], outs[2][0][k]), k
    assert torch.equal(outs[1][1], outs[2][1])
    got = np64(outs[1][1]).reshape(-1, spec.dim)
    check_rows(got, want.reshape(-1, spec.dim))
    assert np.max(np.abs(got - want.reshape(-1, spec.dim))) <= 2e-2
    # the queries alone
    gpu = to_device(cpu)
    step = LayerStep(gpu)
    qo = torch.empty_like(q_raw).cuda()
    dsa.dsa_compress_jobs(step.kind, gpu["cu_new"], gpu["start_pos"], 0, gpu["state_slot"], gpu["state_x"].shape[0],
                          step._jobs(), dev_status=step.status, query=dsa.query_job(q_raw.cuda(), qo, gpu["q_pos"],
                                                                                     step.rope_main))
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    assert torch.equal(qo.cpu(), outs[1][1])


def _oracle_scores_on_gpu_pool(cpu, gpu):
    pool = idx_pool(gpu)
    return OL.index_scores(np64(cpu["q8"]), np64(cpu["q_scale"]), np64(cpu["w"]), np64(cpu["q_pos"]),
                           np64(cpu["q_req"]), pool, np64(cpu["bt_idx"]))


def _check_score_rows(got, want, nvis, gn=None, ld=None):
    """Each query's score row: rel-L2 <= 1e-2 over its visible entries, -inf to the end of their tile."""
    rows_g, rows_w = [], []
    for q, n in nvis.items():
        if gn is not None:
            assert gn[q] == n
        if ld is not None:
            tile_end = min(ld, ((n + 127) // 128) * 128) if n else 0
            assert np.all(np.isneginf(got[q, n:tile_end])), q
        if n:
            rows_g.append(got[q, :n])
            rows_w.append(want[q][:n])
    for j, (g, w) in enumerate(zip(rows_g, rows_w)):
        e = rel_l2(g, w)
        assert e <= ROW_REL_L2, (j, e)


@pytest.mark.parametrize("name", INDEXED)
def test_index_scores(name):
    cpu, gpu, step = _setup(name)
    step.compress()
    step.index()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    want, nvis = _oracle_scores_on_gpu_pool(cpu, gpu)
    _check_score_rows(np64(step.scores), want, nvis, np64(step.n_visible), step.ld)


@pytest.mark.parametrize("name", ["c4a_decode", "c4a_chunk", "c4a_multi_prefill", "c4a_chunk_fp4"])
def test_index_scores_signed_scales(name):
    """Negative query scales in some query groups and negative key scales on some entries: the ReLU
    then keeps the other sign of <q8, k8>, so both the folded-weight path (with its sign branch per
    entry) and the literal formula of groups holding a negative query scale are exercised.  Groups are
    1 (decode), 4 and 32 queries wide."""
    cpu, gpu, step = _setup(name)
    step.compress()
    torch.cuda.synchronize()
    nq, heads = cpu["q_scale"].shape
    qs = cpu["q_scale"].clone()
    flip = torch.zeros_like(qs, dtype=torch.bool)
    flip[: nq // 2 : 3, 1] = True  # a negative head scale in early queries only: later groups stay non-negative
    qs[flip] = -qs[flip]
    gpu["q_scale"].copy_(qs.to(gpu["q_scale"].device))
    ks = gpu["idx_scale"]
    ks[::5] = -ks[::5]  # every fifth physical key row
    step.index()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    pool = idx_pool(gpu)
    want, nvis = OL.index_scores(np64(cpu["q8"]), np64(qs), np64(cpu["w"]), np64(cpu["q_pos"]),
                                 np64(cpu["q_req"]), pool, np64(cpu["bt_idx"]))
    _check_score_rows(np64(step.scores), want, nvis)
    assert any(np.any(want[q][:n] > 0) for q, n in nvis.items())


@pytest.mark.parametrize("name", INDEXED)
def test_topk(name):
    cpu, gpu, step = _setup(name)
    step.compress()
    step.index()
    step.select()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    k = cpu["spec"].topk
    scores, gidx, nv = np64(step.scores), np64(step.topk), np64(step.n_visible)
    for q in range(cpu["nq"]):
        # same fp32 scores -> identical index list (increasing order, -1 padded)
        assert list(gidx[q]) == list(OL.topk(scores[q], int(nv[q]), k))
    want, nvis = _oracle_scores_on_gpu_pool(cpu, gpu)
    for q, n in nvis.items():
        ok, nd = topk_sets_match(gidx[q], want[q], n, k)
        assert ok, (q, nd)


@pytest.mark.parametrize("name", list(CASES))
def test_attention(name):
    cpu, gpu, step = _setup(name)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    spec, epb = cpu["spec"], cpu["epb"]
    main = oracle_pool(gpu["main_data"], gpu["main_scale"], epb)
    swa = oracle_pool(gpu["swa_data"], gpu["swa_scale"], 256)
    topk = np64(step.topk) if step.has_index else None
    want, lse = OL.sparse_attn(np64(cpu["q"]), np64(cpu["q_pos"]), np64(cpu["q_req"]), spec.kind, topk, main,
                               np64(cpu["bt_main"]), swa, np64(cpu["bt_swa"]), spec.window, SM_SCALE, spec.rope_dim)
    got, glse = np64(step.out), np64(step.lse)
    W = np.stack([want[q] for q in range(cpu["nq"])])
    assert_attn_close(got, W, pool_absmax((gpu["main_data"], gpu["main_scale"]), (gpu["swa_data"], gpu["swa_scale"])))
    assert np.max(np.abs(glse - np.stack([lse[q] for q in range(cpu["nq"])]))) <= 1e-3


SELECT_ATTEND = {
    # 32 decode rows of 64 heads: one cluster of four CTAs per row, so the top-k runs inside the attention kernel;
    # ragged contexts, rows below k visible entries (the identity top-k) and rows near the 16,384-score limit
    "c4a_decode_32": S("c4a_decode_32", cached=[int(x) for x in np.random.default_rng(30).integers(100, 65500, 30)]
                       + [1500, 65535], new=[1] * 32, seed=30),
    "c4a_decode_32_fp8": S("c4a_decode_32_fp8", cached=[int(x) for x in np.random.default_rng(31).integers(100, 40000, 32)],
                           new=[1] * 32, main_dtype="fp8", swa_dtype="fp8", seed=31),
}


def _fused_pair(name):
    cpu = synth.make_case(SELECT_ATTEND[name], "cpu")
    gpu = to_device(cpu)
    fused, separate = LayerStep(gpu, fused_select=True), LayerStep(gpu)
    assert fused.fused_select and fused.select_attend_kernels == 1, "the case must run the one-kernel path"
    return cpu, gpu, fused, separate


@pytest.mark.parametrize("name", list(SELECT_ATTEND))
def test_fused_topk_attention_equals_separate_calls(name):
    """The fused call selects exactly the top-k dsa_topk selects and attends exactly as dsa_sparse_attn_decode
    does over it (the same kernel code after the selection): indices, output and lse bit-identical; the output
    also matches the oracle."""
    cpu, gpu, fused, separate = _fused_pair(name)
    separate.run()
    torch.cuda.synchronize()
    t_sep, o_sep, l_sep = separate.topk.clone(), separate.out.clone(), separate.lse.clone()
    fused.run()
    torch.cuda.synchronize()
    assert int(fused.status.item()) == 0 and int(separate.status.item()) == 0
    assert torch.equal(fused.topk, t_sep)
    assert torch.equal(fused.out, o_sep)
    assert torch.equal(fused.lse, l_sep)
    spec, epb = cpu["spec"], cpu["epb"]
    main = oracle_pool(gpu["main_data"], gpu["main_scale"], epb)
    swa = oracle_pool(gpu["swa_data"], gpu["swa_scale"], 256)
    want, lse = OL.sparse_attn(np64(cpu["q"]), np64(cpu["q_pos"]), np64(cpu["q_req"]), spec.kind, np64(fused.topk),
                               main, np64(cpu["bt_main"]), swa, np64(cpu["bt_swa"]), spec.window, SM_SCALE,
                               spec.rope_dim)
    W = np.stack([want[q] for q in range(cpu["nq"])])
    assert_attn_close(np64(fused.out), W, pool_absmax((gpu["main_data"], gpu["main_scale"]),
                                                      (gpu["swa_data"], gpu["swa_scale"])))
    assert np.max(np.abs(np64(fused.lse) - np.stack([lse[q] for q in range(cpu["nq"])]))) <= 1e-3
    # the indices against the oracle's top-k of the same scores
    scores, nv = np64(fused.scores), np64(fused.n_visible)
    for q in range(cpu["nq"]):
        assert list(np64(fused.topk)[q]) == list(OL.topk(scores[q], int(nv[q]), spec.topk)), q


def test_fused_topk_attention_bad_visible_count():
    """A row whose visible count exceeds its score row is a device fault in both forms: its top-k row is all -1,
    its attention sees the window only, and every other row is unchanged."""
    cpu, gpu, fused, separate = _fused_pair("c4a_decode_32")
    bad = 5
    outs = []
    for st in (separate, fused):
        st.compress()
        st.index()
        st.n_visible[bad] = st.ld + 4
        if st is fused:
            st.select_attend()
        else:
            st.select()
            st.attend()
        torch.cuda.synchronize()
        assert int(st.status.item()) == dsa.DSA_ERR_DEVICE_FAULT
        assert bool((st.topk[bad] == -1).all())
        outs.append((st.topk.clone(), st.out.clone(), st.lse.clone()))
    for x, y in zip(*outs):
        assert torch.equal(x, y)


SHARP = {
    # 4 rows: clusters of 4 CTAs and two key splits per row (split partials merged by the combine kernel)
    "c4a_decode": CASES["c4a_decode"],
    # 48 rows: clusters of 2 CTAs
    "c4a_decode_48": S("c4a_decode_48", cached=[int(x) for x in np.random.default_rng(18).integers(600, 3000, 48)],
                       new=[1] * 48, seed=18),
    # dense over c128a entries, a long key list per CTA
    "c128a_decode": CASES["c128a_decode"],
    # 128 query heads: two 64-head groups per row, each its own cluster
    "c4a_decode_128h": S("c4a_decode_128h", cached=[1500, 3071], new=[1, 1], heads=128, seed=19),
}


@pytest.mark.parametrize("name", list(SHARP))
def test_attention_sharp_scores(name):
    """Queries scaled by 40: logits spread over hundreds of log2 units, so a CTA's running maximum
    keeps moving between sub-tiles (the rescale path) and the softmax is nearly one-hot."""
    cpu = synth.make_case(SHARP[name], "cpu")
    gpu = to_device(cpu)
    gpu["q"].mul_(40.0)
    step = LayerStep(gpu)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    spec, epb = cpu["spec"], cpu["epb"]
    main = oracle_pool(gpu["main_data"], gpu["main_scale"], epb)
    swa = oracle_pool(gpu["swa_data"], gpu["swa_scale"], 256)
    topk = np64(step.topk) if step.has_index else None
    want, lse = OL.sparse_attn(np64(gpu["q"]), np64(cpu["q_pos"]), np64(cpu["q_req"]), spec.kind, topk, main,
                               np64(cpu["bt_main"]), swa, np64(cpu["bt_swa"]), spec.window, SM_SCALE, spec.rope_dim)
    got, glse = np64(step.out), np64(step.lse)
    W = np.stack([want[q] for q in range(cpu["nq"])])
    assert_attn_close(got, W, pool_absmax((gpu["main_data"], gpu["main_scale"]), (gpu["swa_data"], gpu["swa_scale"])))
    L = np.stack([lse[q] for q in range(cpu["nq"])])
    assert np.max(np.abs(glse - L) / np.maximum(1.0, np.abs(L))) <= 1e-4


def test_gather_rows_bit_exact_and_unmapped_fault():
    from compressed_sparse_attention_c4a_gb300 import dsa
    cpu, gpu, step = _setup("c4a_decode")
    bt = np64(cpu["bt_main"])
    rng = np.random.default_rng(0)
    req = rng.integers(0, 4, 300).astype(np.int32)
    ids = np.array([rng.integers(0, 64 * int((bt[r] >= 0).sum())) for r in req], dtype=np.int32)
    out = torch.empty((300, 1024), dtype=torch.uint8, device="cuda")
    dsa.dsa_gather_rows(step.main, step.main_bt, torch.from_numpy(req).cuda(), torch.from_numpy(ids).cuda(), out,
                        dev_status=step.status)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    raw = cpu["main_data"].view(torch.uint8).view(-1, 1024).numpy()
    want = raw[[int(bt[r][i // 64]) * 64 + i % 64 for r, i in zip(req, ids)]]
    assert np.array_equal(out.cpu().numpy(), want)
    # a row in an unmapped block: zeros and a device fault status, other rows intact
    bad = torch.tensor([0, 0], dtype=torch.int32, device="cuda")
    bad_ids = torch.tensor([5, 64 * bt.shape[1] - 1], dtype=torch.int32, device="cuda")
    bt_holes = gpu["bt_main"].clone()
    bt_holes[0, -1] = -1
    out2 = torch.full((2, 1024), 7, dtype=torch.uint8, device="cuda")
    dsa.dsa_gather_rows(step.main, dsa.block_table(bt_holes), bad, bad_ids, out2, dev_status=step.status)
    torch.cuda.synchronize()
    assert int(step.status.item()) == dsa.DSA_ERR_DEVICE_FAULT
    assert np.array_equal(out2[0].cpu().numpy(), raw[int(bt[0][0]) * 64 + 5])
    assert int(out2[1].sum().item()) == 0


@pytest.mark.parametrize("ld", [1024, 16384, 20004, 34816, 65536])
def test_topk_edge_cases_exact(ld):
    """Ties, all-equal rows, n == k + 1, n < k, empty rows, -inf tails, negative scores, rows whose
    k-th entry is -inf; rows held in registers (ld <= 16,384), in one CTA's shared memory (up to
    40,960) and split over a cluster (ld > 40,960)."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    rng = np.random.default_rng(ld)
    k = 512
    rows, nv = [], []
    n_full = ld - 3
    for case in range(10):
        r = rng.standard_normal(ld).astype(np.float32)
        n = n_full
        if case == 0:
            r[:] = 1.5                                              # all equal: lowest indices win
        elif case == 1:
            r = rng.integers(0, 7, ld).astype(np.float32)           # heavy ties at the threshold
        elif case == 2:
            n = min(ld, k + 1)
        elif case == 3:
            n = k - 5
        elif case == 4:
            n = 0
        elif case == 5:
            r = -np.abs(r)                                          # negative scores
        elif case == 6:
            r[n_full // 2:] = -np.inf                               # many invisible-looking entries
        elif case == 7:
            r = (rng.integers(0, 3, ld) * 2.0 ** -20).astype(np.float32)   # ties among tiny values
        elif case == 8:
            r[::2] = 0.0                                            # half exact zeros (ReLU-like)
        elif case == 9:
            fin = rng.choice(n_full, 100, replace=False)            # 100 finite scores: the other k - 100
            r[:] = -np.inf                                          # winners are -inf, lowest index first
            r[fin] = rng.standard_normal(100).astype(np.float32)
        rows.append(r)
        nv.append(n)
    scores = torch.from_numpy(np.stack(rows)).cuda()
    n_valid = torch.tensor(nv, dtype=torch.int32, device="cuda")
    out = torch.empty((len(rows), k), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsa.dsa_topk(scores, n_valid, k, out, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().numpy()
    for i, (r, n) in enumerate(zip(rows, nv)):
        assert list(got[i]) == list(OL.topk(r.astype(np.float64), n, k)), i


def test_topk_many_rows_exact():
    """Many rows of random length: random scores, and rows of heavy ties that mix -0 and +0 (equal
    scores: the lower index wins), against the oracle's top-k index for index."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    rng = np.random.default_rng(77)
    nq, ld, k = 700, 4096, 512
    scores = rng.standard_normal((nq, ld)).astype(np.float32)
    scores[::7] = np.round(scores[::7] * 2)                      # heavy ties on every 7th row
    nv = rng.integers(0, ld + 1, nq).astype(np.int32)
    nv[::5] = ld
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((nq, k), dtype=torch.int32, device="cuda")
    dsa.dsa_topk(torch.from_numpy(scores).cuda(), torch.from_numpy(nv).cuda(), k, out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out.cpu().numpy()
    for i in range(nq):
        assert list(got[i]) == list(OL.topk(scores[i].astype(np.float64), int(nv[i]), k)), i


@pytest.mark.parametrize("ld", [1004, 6004, 12292, 16384])
def test_topk_short_rows_on_a_cluster_exact(ld):
    """Few short rows run on a cluster of four CTAs, a quarter of the row each (parts that hold no visible
    score included): random rows, heavy ties across the quarters, rows of one repeated value, and random
    lengths, against the oracle's top-k index for index."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    assert dsa.dsa_topk_plan(40, ld, 512) == (0, 4, 512)
    rng = np.random.default_rng(ld + 1)
    nq, k = 40, 512
    scores = rng.standard_normal((nq, ld)).astype(np.float32)
    scores[1::4] = np.round(scores[1::4] * 3)                    # heavy ties (radix select)
    scores[2::8] = 0.25                                          # one value (take the lowest indices)
    scores[3::8, ld // 2:] = -np.inf
    nv = rng.integers(0, ld + 1, nq).astype(np.int32)
    nv[::3] = ld
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((nq, k), dtype=torch.int32, device="cuda")
    dsa.dsa_topk(torch.from_numpy(scores).cuda(), torch.from_numpy(nv).cuda(), k, out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out.cpu().numpy()
    for i in range(nq):
        assert list(got[i]) == list(OL.topk(scores[i].astype(np.float64), int(nv[i]), k)), i


@pytest.mark.parametrize("nq,ld", [(200, 34816), (120, 20004), (16, 65536)])
def test_topk_long_rows_cluster_sizes_exact(nq, ld):
    """Rows longer than 16,384 scores at row counts that give clusters of 1 (200 rows), 2 (120 rows) and
    4 CTAs per row (16 rows) on 152 SMs: random lengths, ReLU-like zeros and heavy ties, index for index."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    rng = np.random.default_rng(nq + ld)
    k = 512
    scores = np.maximum(rng.standard_normal((nq, ld)), 0.0).astype(np.float32)   # about half exact zeros
    scores[::3] = np.round(scores[::3] * 4) / 4                                     # heavy ties
    nv = rng.integers(k - 10, ld + 1, nq).astype(np.int32)
    nv[::4] = ld
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((nq, k), dtype=torch.int32, device="cuda")
    dsa.dsa_topk(torch.from_numpy(scores).cuda(), torch.from_numpy(nv).cuda(), k, out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out.cpu().numpy()
    for i in range(nq):
        assert list(got[i]) == list(OL.topk(scores[i].astype(np.float64), int(nv[i]), k)), i


@pytest.mark.parametrize("name", ["c4a_decode", "c4a_multi_prefill"])
def test_index_scores_fresh_pos(name):
    """fresh_pos says from which raw position the preceding kernel may still be compressing keys: the
    compressor's own start (the entries before it are scored before the wait), position 0 (every copy
    waits) or past every query (nothing waits) must give the scores of the call without it, bit for bit.
    The entries complete before position p are n_vis(p - 1) = entries i with 4i + 7 < p."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    cpu, gpu, step = _setup(name)
    step.compress()
    torch.cuda.synchronize()
    c = step.case
    runs = []
    batch = cpu["spec"].batch
    for fresh in (None, torch.zeros(batch, dtype=torch.int32, device="cuda"),
                  torch.full((batch,), 1 << 30, dtype=torch.int32, device="cuda"), c["start_pos"]):
        scores = torch.full_like(step.scores, float("nan"))
        dsa.dsa_index_scores(c["q8"], c["q_scale"], c["w"], c["q_pos"], c["q_req"], step.q_group, step.idx,
                             step.idx_bt, scores, step.n_visible, dev_status=step.status, fresh_pos=fresh)
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0
        runs.append(np64(scores))
    nv = np64(step.n_visible)
    for q in range(cpu["nq"]):
        n = int(nv[q])
        assert np.array_equal(runs[1][q, :n], runs[0][q, :n]), q
        assert np.array_equal(runs[2][q, :n], runs[0][q, :n]), q
        assert np.array_equal(runs[3][q, :n], runs[0][q, :n]), q


@pytest.mark.parametrize("name", ["c4a_decode", "c4a_multi_prefill", "c4a_decode_fp4", "c4a_chunk"])
def test_index_work_counter_same_scores_and_left_zero(name):
    """With a work counter the CTAs take runs of items dynamically: the scores equal those of the static
    split bit for bit, and each call leaves the counter zero (three calls in a row)."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    cpu, gpu, step = _setup(name)
    step.compress()
    torch.cuda.synchronize()
    c = step.case
    work = torch.zeros((4,), dtype=torch.int32, device="cuda")
    runs = []
    for wk in (None, work, work, work):
        scores = torch.full_like(step.scores, float("nan"))
        dsa.dsa_index_scores(c["q8"], c["q_scale"], c["w"], c["q_pos"], c["q_req"], step.q_group, step.idx,
                             step.idx_bt, scores, step.n_visible, dev_status=step.status, fresh_pos=step.fresh_pos,
                             work=wk)
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0
        assert int(work.count_nonzero().item()) == 0
        runs.append(np64(scores))
    nv = np64(step.n_visible)
    for q in range(cpu["nq"]):
        n = int(nv[q])
        for r in runs[1:]:
            assert np.array_equal(r[q, :n], runs[0][q, :n]), q


# ---- device-detected faults: a needed block unmapped (-1) in one request's table ---------------------
# Every kernel resolves its paged reads and writes through the checked block-table translation; an unmapped
# block raises DSA_ERR_DEVICE_FAULT and affects only the rows that needed it.

def test_compress_unmapped_block_faults_only_that_entry():
    from compressed_sparse_attention_c4a_gb300 import dsa
    cpu, gpu, step = _setup("c4a_decode")          # new tokens 1000, 2999, 777, 4095: 2999 and 4095 close entries
    r, i = 1, (2999 - 7) // 4                        # request 1's new entry 748, block 11 of its main table
    prow = int(gpu["bt_main"][r, i // 64]) * 64 + i % 64
    before = gpu["main_data"][prow].clone()
    gpu["bt_main"][r, i // 64] = -1
    step.compress()
    torch.cuda.synchronize()
    assert int(step.status.item()) == dsa.DSA_ERR_DEVICE_FAULT
    assert torch.equal(gpu["main_data"][prow], before)           # the unmapped entry is not written anywhere
    rec = {}
    pool, swa, states, emitted = _oracle_compress(cpu, "main", rec)
    assert emitted[1] == [i] and emitted[3] == [(4095 - 7) // 4]
    bt = np64(cpu["bt_main"])
    j = emitted[3][0]
    check_pool_rows(gpu["main_data"], gpu["main_scale"], [int(bt[3][j // 64]) * 64 + j % 64], [rec[("entry", 3, j)]],
                    [pool.read(bt[3], [j])[0]])
    sbt = np64(cpu["bt_swa"])
    start = np64(cpu["start_pos"])
    prows = [int(sbt[q][int(start[q]) // 256]) * 256 + int(start[q]) % 256 for q in range(4)]
    check_pool_rows(gpu["swa_data"], gpu["swa_scale"], prows, [rec[("swa", q, int(start[q]))] for q in range(4)],
                    [swa.read(sbt[q], [int(start[q])])[0] for q in range(4)])


@pytest.mark.parametrize("counted,name", [(False, "c4a_decode"), (True, "c4a_decode"), (False, "c4a_decode_fp4")])
def test_index_unmapped_block_scores_minus_inf(counted, name):
    """Plain indexer + top-k, and the indexer that counts the top-k's first digit + the top-k from the counts;
    e4m3 and e2m1 keys."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    cpu = synth.make_case(CASES[name], "cpu")
    gpu = to_device(cpu)
    step = LayerStep(gpu, counted_topk=counted)
    assert step.fused_topk == counted
    step.compress()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    want, nvis = _oracle_scores_on_gpu_pool(cpu, gpu)     # with the intact table
    r, lb = 2, 1                                         # request 2 (193 visible entries): entries 64 .. 127
    gpu["bt_idx"][r, lb] = -1
    step.index()
    step.select()
    torch.cuda.synchronize()
    assert int(step.status.item()) == dsa.DSA_ERR_DEVICE_FAULT
    got = np64(step.scores)
    assert nvis[r] == 193
    assert np.all(np.isneginf(got[r, 64:128]))
    keep = np.r_[0:64, 128:193]
    assert rel_l2(got[r, keep], want[r][keep]) <= ROW_REL_L2
    _check_score_rows(got, want, {q: n for q, n in nvis.items() if q != r})
    tk, nv = np64(step.topk), np64(step.n_visible)        # the counted top-k sees the -inf entries as scores
    for q in range(cpu["nq"]):
        assert list(tk[q]) == list(OL.topk(got[q], int(nv[q]), cpu["spec"].topk)), q
    if counted:
        assert int(step.topk_ws.count_nonzero().item()) == 0


@pytest.mark.parametrize("wait_ms,name", [(20, "c4a_decode"), (20, "c4a_multi_prefill")])
def test_index_bounded_wait_expires_then_next_call_is_correct(wait_ms, name):
    """The indexer with its copies withheld: every consumer wait runs out after the given limit, the kernel
    records DSA_ERR_TIMEOUT, frees its tensor memory and returns; the next normal call is correct."""
    import time
    from compressed_sparse_attention_c4a_gb300 import dsa
    cpu, gpu, step = _setup(name)
    step.compress()
    torch.cuda.synchronize()
    c = step.case
    scores = torch.full_like(step.scores, float("nan"))
    t0 = time.time()
    dsa.dsa_debug_index_scores_stalled(c["q8"], c["q_scale"], c["w"], c["q_pos"], c["q_req"], step.q_group, step.idx,
                                       step.idx_bt, scores, wait_ms * 1_000_000, n_visible=step.n_visible,
                                       dev_status=step.status)
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert int(step.status.item()) == dsa.DSA_ERR_TIMEOUT
    assert bool(torch.isnan(scores).all())                       # nothing was scored
    step.status.zero_()
    step.index()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    want, nvis = _oracle_scores_on_gpu_pool(cpu, gpu)
    _check_score_rows(np64(step.scores), want, nvis, np64(step.n_visible), step.ld)


@pytest.mark.parametrize("name", ["c4a_decode", "c4a_decode_48"])
def test_attention_unmapped_block_zeroes_the_row(name):
    """A selected entry in an unmapped main block (one row) and an unmapped window block (another row): both
    rows are written as zeros with lse = -inf, the others still match the oracle.  Four rows split their keys
    over two clusters (the partials' merge kernel zeroes the row); 48 rows merge inside one cluster."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    spec = CASES.get(name) or SHARP[name]
    cpu = synth.make_case(spec, "cpu")
    gpu = to_device(cpu)
    step = LayerStep(gpu)
    step.compress()
    step.index()
    step.select()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    tk = np64(step.topk)
    bt_main0, bt_swa0 = np64(cpu["bt_main"]), np64(cpu["bt_swa"])
    ra, rb = 0, 3
    ida = int(tk[ra][tk[ra] >= 0][len(tk[ra][tk[ra] >= 0]) // 2])
    gpu["bt_main"][ra, ida // 64] = -1
    mb = int(np64(cpu["q_pos"])[rb])
    gpu["bt_swa"][rb, mb // 256] = -1                     # the block of row rb's own position
    step.attend()
    torch.cuda.synchronize()
    assert int(step.status.item()) == dsa.DSA_ERR_DEVICE_FAULT
    out, lse = np64(step.out), np64(step.lse)
    for r in (ra, rb):
        assert np.all(out[r] == 0.0), r
        assert np.all(np.isneginf(lse[r])), r
    main = oracle_pool(gpu["main_data"], gpu["main_scale"], cpu["epb"])
    swa = oracle_pool(gpu["swa_data"], gpu["swa_scale"], 256)
    rows = [q for q in range(cpu["nq"]) if q not in (ra, rb)]
    want, wl = OL.sparse_attn(np64(cpu["q"]), np64(cpu["q_pos"]), np64(cpu["q_req"]), spec.kind, tk, main, bt_main0,
                              swa, bt_swa0, spec.window, SM_SCALE, spec.rope_dim, rows=rows)
    W = np.stack([want[q] for q in rows])
    assert_attn_close(out[rows], W, pool_absmax((gpu["main_data"], gpu["main_scale"]), (gpu["swa_data"], gpu["swa_scale"])))
    assert np.max(np.abs(lse[rows] - np.stack([wl[q] for q in rows]))) <= 1e-3



# ---- indexer with the top-k's first digit counted while scoring, and the top-k that starts from it ---------
FUSED = {
    "c4a_decode": CASES["c4a_decode"],                 # four rows, one of them below k
    "c4a_decode_48": SHARP["c4a_decode_48"],           # 48 rows, each spread over several CTAs
    "c4a_multi_prefill": CASES["c4a_multi_prefill"],   # groups of 32 queries selected by the CTA finishing them
    "c4a_early": CASES["c4a_early"],                   # groups of 4; rows without a visible entry
}


def _fused_call(step, ws, idx):
    from compressed_sparse_attention_c4a_gb300 import dsa
    c = step.case
    dsa.dsa_index_topk(c["q8"], c["q_scale"], c["w"], c["q_pos"], c["q_req"], step.q_group, step.idx, step.idx_bt,
                       step.scores, step.spec.topk, idx, ws, step.n_visible, dev_status=step.status,
                       fresh_pos=step.fresh_pos)


@pytest.mark.parametrize("name", list(FUSED))
def test_index_topk_fused_exact(name):
    """dsa_index_topk (the indexer counting each row's first radix digit, then the top-k starting from those
    counts) lists, for the very scores it wrote, exactly the indices the oracle's top-k takes (ties to the lower
    index, increasing order, -1 padding); twice in a row, the counts back to zero each time."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    spec = FUSED[name]
    cpu = synth.make_case(spec, "cpu")
    gpu = to_device(cpu)
    step = LayerStep(gpu)
    step.compress()
    torch.cuda.synchronize()
    nq, k = cpu["nq"], spec.topk
    ws = torch.zeros((dsa.dsa_index_topk_workspace_size(nq),), dtype=torch.uint8, device="cuda")
    want, nvis = _oracle_scores_on_gpu_pool(cpu, gpu)
    for _ in range(2):
        idx = torch.full((nq, k), -7, dtype=torch.int32, device="cuda")
        step.scores.fill_(float("nan"))
        _fused_call(step, ws, idx)
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0
        assert int(ws.count_nonzero().item()) == 0
        got, gi, nv = np64(step.scores), np64(idx), np64(step.n_visible)
        _check_score_rows(got, want, nvis, nv, step.ld)
        for q in range(nq):
            assert list(gi[q]) == list(OL.topk(got[q], int(nv[q]), k)), q
            ok, nd = topk_sets_match(gi[q], want[q], int(nv[q]), k)
            assert ok, (q, nd)


def test_index_topk_fused_heavy_ties():
    """Rows whose scores are all equal (one request's key rows all the same; another request's head weights
    all zero, so every score is 0): the selection descends to the exact tied key and takes the lowest indices."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    cpu, gpu, step = _setup("c4a_decode")
    step.compress()
    torch.cuda.synchronize()
    bt = gpu["bt_idx"]
    r = 3                                                  # m = 4095: 1023 visible entries in blocks 0 .. 15
    src = int(bt[r, 0]) * 64
    for lb in range(16):
        pb = int(bt[r, lb])
        gpu["idx_data"][pb * 64:(pb + 1) * 64] = gpu["idx_data"][src]
        gpu["idx_scale"][pb * 64:(pb + 1) * 64] = gpu["idx_scale"][src]
    gpu["w"][1].zero_()                                     # request 1 (749 visible entries): every score 0
    ws = torch.zeros((dsa.dsa_index_topk_workspace_size(cpu["nq"]),), dtype=torch.uint8, device="cuda")
    idx = torch.full((cpu["nq"], 512), -7, dtype=torch.int32, device="cuda")
    _fused_call(step, ws, idx)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    gi, got, nv = np64(idx), np64(step.scores), np64(step.n_visible)
    assert np.all(got[3, :1023] == got[3, 0]) and np.all(got[1, :749] == 0.0)
    assert list(gi[3]) == list(range(512)) and list(gi[1]) == list(range(512))
    for q in range(cpu["nq"]):
        assert list(gi[q]) == list(OL.topk(got[q], int(nv[q]), 512)), q
    assert int(ws.count_nonzero().item()) == 0


# ---- fp8 attention output (inverse RoPE + fp8 quantisation in one pass) ------------------------------------
Q8_CASES = {
    "c4a_decode": CASES["c4a_decode"],          # keys split over two clusters: the partials' merge kernel quantises
    "c4a_decode_48": SHARP["c4a_decode_48"],    # clusters of two CTAs: the owners quantise their tiles
    "c4a_chunk": CASES["c4a_chunk"],            # one CTA per row: four tiles in turn
    "c128a_decode": CASES["c128a_decode"],
}


@pytest.mark.parametrize("name", list(Q8_CASES))
def test_attention_fp8_output(name):
    """dsa_sparse_attn_q8 against (a) the oracle's float64 output, within the attention tolerance plus half an
    e4m3 step, and (b) the same kernel's bf16 output: each block's scale is the amax / 448 of those values, each
    code a correct rounding of value / scale (a code decides an integer from a float: the slack covers only the
    bf16 rounding of the reference values); lse as the bf16 call's."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    from _parity import fp8_row_violations
    from oracle.codecs import e4m3_decode
    spec = Q8_CASES[name]
    cpu = synth.make_case(spec, "cpu")
    gpu = to_device(cpu)
    step = LayerStep(gpu)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    nq, H = cpu["nq"], spec.heads
    codes = torch.full((nq, H, 512), 0x7F, dtype=torch.uint8, device="cuda")
    scale = torch.full((nq, H, 4), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.empty((nq, H), dtype=torch.float32, device="cuda")
    tk = step.topk if step.has_index else None
    c = step.case
    dsa.dsa_sparse_attn_q8(c["q"], c["q_pos"], c["q_req"] if spec.queries == "all" else None, step.kind, tk,
                           spec.topk if step.has_index else 0, step.main, step.main_bt, step.swa, step.swa_bt,
                           spec.window, SM_SCALE, step.rope_main, codes, scale, lse, step.workspace,
                           dev_status=step.status)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    cg, sg = codes.cpu().numpy(), np64(scale)
    deq = (e4m3_decode(cg).reshape(nq, H, 4, 128) * sg[..., None]).reshape(nq, H, 512)
    main = oracle_pool(gpu["main_data"], gpu["main_scale"], cpu["epb"])
    swa = oracle_pool(gpu["swa_data"], gpu["swa_scale"], 256)
    want, wl = OL.sparse_attn(np64(cpu["q"]), np64(cpu["q_pos"]), np64(cpu["q_req"]), spec.kind,
                              np64(step.topk) if step.has_index else None, main, np64(cpu["bt_main"]), swa,
                              np64(cpu["bt_swa"]), spec.window, SM_SCALE, spec.rope_dim)
    W = np.stack([want[q] for q in range(nq)])
    vmax = pool_absmax((gpu["main_data"], gpu["main_scale"]), (gpu["swa_data"], gpu["swa_scale"]))
    bound = np.abs(W) * 2.0 ** -4 + np.repeat(sg, 128, axis=-1) * 2.0 ** -10 + attn_bound(W, vmax)
    assert np.all(np.abs(deq - W) <= bound)
    for q in range(nq):
        assert rel_l2(deq[q], W[q]) <= 2.0 ** -4 + ATTN_REL_L2, q
    # the same kernel's bf16 values decide the codes
    ref = np64(step.out).reshape(-1, 128)
    bad_el, bad_rows = fp8_row_violations(cg.reshape(-1, 128), sg.reshape(-1), ref, value_slack=2.0 ** -8,
                                          scale_rel=2.0 ** -8)
    assert len(bad_rows) == 0, bad_rows[:8]
    assert len(bad_el) == 0, bad_el[:8]
    assert np.allclose(np64(lse), np64(step.lse), rtol=0, atol=1e-6)

"""build_k2q_csr + schedule on the GPU, bit-exact against the oracle's CSR
(plain loops) and its work-list rule (vLLM docs, sparse_attention_msa,
MiniMaxM3SparseMSAImpl.forward: build_k2q_csr over [H, T, 16] page lists,
total_rows = total_kv_blocks)."""
import numpy as np
import pytest
import torch

import block_sparse_attention_prefill_gb300 as msa
import oracle
import pins
import workloads

pytestmark = pytest.mark.gpu


def gpu_plan(w, total_rows=None):
    wd = w.to("cuda")
    R = w.total_rows if total_rows is None else total_rows
    plan = msa.msa_plan(wd.topk, wd.cu_q, wd.cu_k, wd.block_table,
                        w.num_pages, w.Hq, R, max(w.max_seqlen_q, 1),
                        max(w.max_seqlen_k, 1))
    torch.cuda.synchronize()
    nnz, nwork = plan.counters()
    return plan, nnz, nwork


def compare_plan(w, total_rows=None):
    plan, nnz, nwork = gpu_plan(w, total_rows)
    R = w.total_rows if total_rows is None else total_rows
    check_plan(plan, nnz, nwork, w, R)
    return plan


def check_plan(plan, nnz, nwork, w, R):
    """The GPU plan against the oracle's CSR (plain loops) and its work-list
    rule, bit for bit, plus the attention kernel's records."""
    row_ptr, q_idx, slot, mask = oracle.k2q_csr(w, total_rows=R)
    assert nnz == len(q_idx)
    assert np.array_equal(plan.row_ptr().cpu().numpy(), row_ptr)
    assert np.array_equal(plan.q_idx()[:nnz].cpu().numpy(), q_idx)
    assert np.array_equal(plan.slot()[:nnz].cpu().numpy(), slot)
    got_mask = plan.slot_mask().cpu().numpy().view(np.uint16).reshape(
        mask.shape)
    assert np.array_equal(got_mask, mask)
    items = oracle.schedule(row_ptr, w, total_rows=R)
    assert nwork == len(items)
    work = plan.work()[:nwork].cpu().numpy()
    got = [(int(a), int(b), int(c), int(d) >> 24, int(d) & 0xFFFFFF)
           for a, b, c, d in work]
    assert got == items
    # the attention kernel's records: header {KV row, n, first key, first
    # query head} and per token {t, position, slot}
    recs = plan.records()[:nwork].cpu().numpy()
    bt = w.block_table.numpy()
    cu_q = w.cu_q.numpy()
    G = w.G
    for wi, (start, n, b, h, pg) in enumerate(items):
        hdr = recs[wi, 0]
        phys = int(bt[b, pg])
        assert list(hdr) == [(phys * w.Hkv + h) * 128, n, pg * 128, h * G], wi
        for k in range(n):
            t = int(q_idx[start + k])
            pos = w.seq_lens[b] - w.q_lens[b] + (t - int(cu_q[b]))
            assert list(recs[wi, 1 + k, :3]) == [t, pos, int(slot[start + k])]


@pytest.mark.parametrize("name", ["tiny_full_prefill", "chunked_prefill_32k",
                                  "ragged_batch_8"])
def test_plan_matches_oracle(name):
    w = workloads.make_config(name, seed=0)
    plan = compare_plan(w)
    assert plan.status() == 0


@pytest.mark.parametrize("seed", [3, 4])
def test_plan_invalid_entries(seed):
    w = pins.tiny_sparse_workload(seed)
    plan = compare_plan(w)
    st = plan.status()
    assert st & msa.STATUS_BAD_PAGE_ID
    assert st & msa.STATUS_BAD_BLOCK


def test_plan_group_sizes():
    for hq, hkv in ((16, 1), (12, 4), (8, 8), (128, 1)):
        w = workloads.make_batch("g", [300, 40], [2000, 900], hq, hkv, seed=hq)
        compare_plan(w)


def test_plan_long_rows():
    # a prefill from empty cache: page 0 is selected by thousands of tokens
    w = workloads.make_batch("ctx0", [8192], [8192], 16, 1, seed=1)
    compare_plan(w)


def test_plan_decode_shape_and_spare_rows():
    sl = workloads.decode_lengths(0, 16, 4096, 20000)
    w = workloads.make_batch("dec", [8] * 16, sl, 16, 2, seed=2)
    compare_plan(w, total_rows=w.total_rows + 37)


def test_plan_all_padding_and_empty_requests():
    w = workloads.make_batch("pad", [64, 0, 32], [5000, 300, 32], 8, 2, seed=5)
    w = pins._replace(w, topk=torch.full_like(w.topk, -1))
    plan, nnz, nwork = gpu_plan(w)
    assert nnz == 0 and nwork == 0 and plan.status() == 0
    w2 = workloads.make_batch("pad2", [64, 0, 32], [5000, 300, 32], 8, 2, seed=5)
    compare_plan(w2)


def _early_read_plan(w):
    """True when the plan's bitmap has at least 32 bytes per top-k entry:
    then mark and scatter read their inputs before their dependent-launch
    wait (the library's switch, restated)."""
    W = 4 * -(-w.max_seqlen_q // 128)
    return w.Hkv * w.total_rows * W * 4 >= 32 * w.T * w.Hkv * 16


@pytest.mark.parametrize("seed", [0, 1])
def test_early_read_plan_with_invalid_entries(seed):
    # few tokens over long contexts (43 bitmap bytes per entry: the early
    # reads), with ids past the request's pages, ids below -1, repeats, a
    # future page and a block_table entry outside the pool, as in the
    # oracle's own pins
    w = workloads.make_batch("early_bad", [150, 12], [300000, 150000], 8, 2, seed=30 + seed)
    assert _early_read_plan(w)
    tk = w.topk.clone()
    tk[0, 0, 5] = 10**6                # past the request's 2344 pages
    tk[1, 1, 3] = -7                   # below -1
    tk[2, 0, 7] = tk[2, 0, 1]          # a repeat
    tk[20, 1, 2] = tk[20, 1, 9]        # a repeat
    tk[155, 0, 4] = 2000               # past request 1's 1172 pages
    tk[0, 1, 8] = 2343                 # token 0 sits on page 2342: a future page
    bt = w.block_table.clone()
    bt[0, int(w.topk[4, 0, 6])] = -1   # a page token 4 selects: not in the pool
    w = pins._replace(w, topk=tk, block_table=bt)
    plan = compare_plan(w)
    st = plan.status()
    assert st & msa.STATUS_BAD_PAGE_ID and st & msa.STATUS_BAD_BLOCK


def test_plan_bad_seqlens_gives_empty_plan():
    w = workloads.make_batch("bad", [64], [5000], 8, 2, seed=6)
    cu_k = w.cu_k.clone()
    cu_k[1] = 30                       # seq_len < q_len
    w = pins._replace(w, cu_k=cu_k)
    plan, nnz, nwork = gpu_plan(w, total_rows=64)
    assert nnz == 0 and nwork == 0
    assert plan.status() & msa.STATUS_BAD_SEQLENS


def test_plan_rows_overflow():
    w = workloads.make_batch("ovf", [16], [5000], 8, 2, seed=7)
    plan, nnz, nwork = gpu_plan(w, total_rows=10)
    assert nnz == 0 and plan.status() & msa.STATUS_ROWS_OVERFLOW


def test_plan_is_deterministic():
    w = workloads.make_config("chunked_prefill_32k", seed=1)
    p1, n1, _ = gpu_plan(w)
    a = p1.q_idx()[:n1].clone()
    for _ in range(3):
        p2, n2, _ = gpu_plan(w)
        assert n2 == n1 and torch.equal(p2.q_idx()[:n2], a)


@pytest.mark.parametrize("name", ["long_prefill_1m", "long_prefill_150k"])
def test_plan_full_size(name):
    # the bench's workloads: 16,384 rows with ~4 tokens each (1M), and
    # 2,400 rows of up to hundreds of tokens (150K)
    w = workloads.make_config(name, seed=0)
    plan = compare_plan(w)
    assert plan.status() == 0


def test_decode_plan_over_65535_rows():
    # msa_decode's plan for 64 requests x 8 tokens over contexts up to 131,072
    # tokens: 2 x 64 x 1024 = 131,072 rows, more than a grid's y or z extent
    # could hold (vLLM PR 64631, Details: page counts go on grid x); checked
    # bit for bit like every other plan
    w = workloads.make_config("decode_64x8", seed=0, kv_device="cuda")
    wd = w.to("cuda")
    n = w.q_lens[0]
    seq = torch.tensor(w.seq_lens, dtype=torch.int32, device="cuda")
    out, lse, plan = msa.msa_decode(wd.q, wd.kv, w.q_scale, w.k_scale,
                                    w.v_scale, w.softmax_scale, wd.topk,
                                    wd.block_table, seq, n, w.max_seqlen_k)
    torch.cuda.synchronize()
    R = int(plan.struct.total_rows)
    assert w.Hkv * R > 65535
    nnz, nwork = plan.counters()
    check_plan(plan, nnz, nwork, w, R)
    assert plan.status() == 0


@pytest.mark.parametrize("hq,q_lens,seq_lens", [
    (16, [100, 30], [1000, 300]),      # 8 + 3 = 11 rows
    (8, [200, 7, 50], [3000, 7, 500]),  # 24 + 1 + 4 = 29 rows
])
def test_plan_odd_row_counts(hq, q_lens, seq_lens):
    # one KV head and an odd number of pages: the last row tile ends inside
    # a warp (two rows per warp, a half-warp each)
    w = workloads.make_batch("odd", q_lens, seq_lens, hq, 1, seed=9)
    assert (w.Hkv * w.total_rows) % 2 == 1
    compare_plan(w)


@pytest.mark.parametrize("q_lens,seq_lens", [
    ([100, 7], [900, 7]),            # 4 words a row: one lane per row
    ([200, 30], [1500, 300]),        # 8 words: two lanes
    ([300, 5], [2600, 500]),         # 12 words: four lanes, one idle
    ([600, 64], [3000, 640]),        # 20 words: eight lanes, three idle
    ([1500, 9], [6000, 900]),        # 48 words: sixteen lanes, four idle
    ([2100, 33], [7000, 3000]),      # 68 words: two vectors a lane, ragged
])
@pytest.mark.parametrize("spare", [0, 300])
def test_plan_row_widths(q_lens, seq_lens, spare):
    # the rows kernel gives a row 1 to 16 lanes by its width (the longest
    # query chunk sets the words per row); odd row counts end a tile inside
    # a round, and spare rows past the pages make several tiles
    w = workloads.make_batch("width", q_lens, seq_lens, 8, 1, seed=len(q_lens) + q_lens[0])
    assert (w.Hkv * (w.total_rows + spare)) % 2 == 1
    compare_plan(w, total_rows=w.total_rows + spare)


@pytest.mark.parametrize("q_len,seq_len,rows", [
    (2048, 300000, 12000),   # 64 words a row, tiles of 6 rounds of 16 rows
    (4096, 40000, 9000),     # 128 words, two vectors a lane, 5 rounds
    (2048, 300000, 70000),   # 560-row tiles: a 512-row segment, then 48 rows
])
def test_plan_tiles_of_many_rounds(q_len, seq_len, rows):
    # spare rows past the last request's pages make the tiles several rounds
    # deep, more than one group of rounds whose loads go out together
    w = workloads.make_batch("deep", [q_len], [seq_len], 16, 2, seed=q_len)
    compare_plan(w, total_rows=rows)


def test_plan_tiles_of_several_segments():
    # 2 x 70,000 rows of one lane: 256 tiles of 768 rows, each worked as a
    # 512-row segment and a 256-row one
    sl = workloads.decode_lengths(3, 16, 4096, 20000)
    w = workloads.make_batch("dec", [8] * 16, sl, 16, 2, seed=11)
    compare_plan(w, total_rows=70000)

"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs.

Small configurations are compared element by element (every cache row, every
logit); the full-size drafters are compared on sampled steps, sequences and
cache rows, which the oracle computes exactly (ingest is row-wise and the
draft steps are open-loop, so any step can be checked on its own).
Tolerances: logits and cache rows max|d| <= 2e-2 * max|ref| in bf16 and
1e-4 * max|ref| in fp32; tokens exactly wherever the oracle's top-2 margin
exceeds that tolerance, otherwise one of the oracle's near-tied chains.
"""
import numpy as np
import pytest

import oracle
import synthetic as syn
from helpers import (check_block, check_cache, make_gpu_drafter, rel_tol, tensor_to_f64, to_torch,
                     weights_to_device)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="session", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_draft_model_gb300 as bdm
    bdm.build()
    bdm.load()


def _draft(gdr, cfg, anchor, want_logits=True):
    tok = torch.empty(cfg.gamma, dtype=torch.int32, device="cuda")
    conf = torch.empty(cfg.gamma, dtype=torch.float32, device="cuda")
    lg = torch.empty(cfg.gamma, cfg.vocab, dtype=torch.float32, device="cuda") if want_logits else None
    gdr.draft(anchor, tok, conf, lg)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), conf.cpu().numpy(), (lg.cpu().numpy() if want_logits else None)


def _small(cfg, L, seed, chunks, anchors, norm_std=0.1, max_ctx=None, paths=()):
    """Ingest L rows in `chunks`, compare every cache row, then draft each anchor and compare.
    paths: (what, value) pairs given to set_path first (which form of the computation runs)."""
    W = syn.make_weights(cfg, seed=seed, norm_std=norm_std)
    X = syn.make_feats(cfg, L, seed=seed)
    dr = oracle.Drafter(cfg, W)
    dr.ingest(X)
    gdr = make_gpu_drafter(cfg, weights_to_device(W), max_ctx=max_ctx or L + 8)
    for what, value in paths:
        gdr.set_path(what, value)
    Xd = to_torch(X)
    lo = 0
    for hi in chunks + [L]:
        gdr.ingest_context(Xd[lo:hi])
        lo = hi
    assert gdr.context_length() == L
    rel = rel_tol(cfg)
    if L:
        check_cache(dr, gdr, cfg, 0, np.arange(L), rel, label="cache")
    for a in anchors:
        tok, conf, lg = _draft(gdr, cfg, a)
        check_block(dr, 0, a, tok, conf, lg, rel=rel, label=f"anchor {a}")
    assert gdr.check() == 0
    return dr, gdr, W


def test_tiny_fp32_drafter():
    """4 heads of 32, 2 layers, gamma 4, V 1024, r 32, 64 context rows, fp32 (1e-4)."""
    cfg = syn.WORKLOADS["tiny_fp32"].cfg
    _small(cfg, 64, seed=0, chunks=[5, 6, 40], anchors=[0, 17, 1023], norm_std=0.0)


def test_tiny_fp32_random_norms_gelu():
    cfg = syn.DrafterConfig(**{**syn.WORKLOADS["tiny_fp32"].cfg.__dict__, "act": "gelu_tanh"})
    _small(cfg, 64, seed=1, chunks=[33], anchors=[5, 900])


def test_bf16_ragged_multi_tile():
    """Shapes that are not multiples of the tiles: d 192 (3 heads of 64), F 384,
    m*H 960, V 1000, r 24, gamma 5, 77 + 3 context rows, random norm weights."""
    cfg = syn.DrafterConfig(hidden=320, n_taps=3, d_draft=192, n_heads=3, n_layers=2, ff_mult=2, gamma=5,
                            vocab=1000, markov_rank=24)
    _small(cfg, 80, seed=2, chunks=[77], anchors=[0, 999, 321])


def test_bf16_single_position_and_empty_context():
    """gamma = 1 (no mask rows) and a draft with no context at all."""
    cfg = syn.DrafterConfig(hidden=128, n_taps=2, d_draft=128, n_heads=2, n_layers=2, ff_mult=2, gamma=1,
                            vocab=512, markov_rank=16)
    W = syn.make_weights(cfg, seed=3, norm_std=0.1)
    dr = oracle.Drafter(cfg, W)
    gdr = make_gpu_drafter(cfg, weights_to_device(W), max_ctx=32)
    tok, conf, lg = _draft(gdr, cfg, 7)
    check_block(dr, 0, 7, tok, conf, lg, label="empty context")
    X = syn.make_feats(cfg, 3, seed=3)
    dr.ingest(X)
    gdr.ingest_context(to_torch(X))
    tok, conf, lg = _draft(gdr, cfg, 8)
    check_block(dr, 0, 8, tok, conf, lg, label="3 rows")


def test_chunked_ingest_matches_one_shot_on_gpu():
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=128, n_heads=2, n_layers=2, ff_mult=2, gamma=4,
                            vocab=640, markov_rank=16)
    W = syn.make_weights(cfg, seed=4)
    Wd = weights_to_device(W)
    X = to_torch(syn.make_feats(cfg, 50, seed=4))
    a = make_gpu_drafter(cfg, Wd, max_ctx=64)
    a.ingest_context(X)
    b = make_gpu_drafter(cfg, Wd, max_ctx=64)
    for lo, hi in ((0, 3), (3, 20), (20, 50)):
        b.ingest_context(X[lo:hi])
    for i in range(cfg.n_layers):
        ka, va = a.cache(0, i, 50)
        kb, vb = b.cache(0, i, 50)
        # different kernels may serve different chunk sizes: compare within the bf16 tolerance
        assert (ka.float() - kb.float()).abs().max().item() <= 2e-2 * ka.float().abs().max().item()
        assert (va.float() - vb.float()).abs().max().item() <= 2e-2 * va.float().abs().max().item()


def test_host_buffer_calls_match_device_calls():
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=128, n_heads=2, n_layers=1, ff_mult=2, gamma=3,
                            vocab=700, markov_rank=16)
    W = syn.make_weights(cfg, seed=5)
    Wd = weights_to_device(W)
    X = syn.make_feats(cfg, 20, seed=5)
    a = make_gpu_drafter(cfg, Wd, max_ctx=32)
    a.ingest_context(to_torch(X))
    ta, ca, la = _draft(a, cfg, 11)
    b = make_gpu_drafter(cfg, Wd, max_ctx=32)
    Xh = torch.from_numpy(X.view(np.int16)).pin_memory()
    b.ingest_context_host(Xh)
    Xh.zero_()  # the call returns once the features have been read: reusing the buffer changes nothing
    tb = torch.empty(cfg.gamma, dtype=torch.int32).pin_memory()
    cb = torch.empty(cfg.gamma, dtype=torch.float32).pin_memory()
    lb = torch.empty(cfg.gamma, cfg.vocab, dtype=torch.float32).pin_memory()
    b.draft_host(11, tb, cb, lb)
    assert np.array_equal(ta, tb.numpy())
    assert np.array_equal(ca, cb.numpy())
    assert np.array_equal(la, lb.numpy())


def test_batched_equals_per_sequence():
    """Three sequences through the batched calls == each sequence on its own handle."""
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=128, n_heads=4, n_layers=2, ff_mult=2, gamma=4,
                            vocab=777, markov_rank=32)
    W = syn.make_weights(cfg, seed=6, norm_std=0.1)
    Wd = weights_to_device(W)
    lens = [9, 0, 23]
    feats = [syn.make_feats(cfg, n, seed=6, seq=i) for i, n in enumerate(lens)]
    gb = make_gpu_drafter(cfg, Wd, max_ctx=40, max_seqs=5)
    ids = torch.tensor([4, 1, 2], dtype=torch.int32, device="cuda")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    allx = to_torch(np.concatenate(feats, axis=0))
    gb.ingest_context_batched(ids, cu, allx)
    anchors = torch.tensor([3, 500, 776], dtype=torch.int32, device="cuda")
    tok = torch.empty(3, cfg.gamma, dtype=torch.int32, device="cuda")
    conf = torch.empty(3, cfg.gamma, dtype=torch.float32, device="cuda")
    lg = torch.empty(3, cfg.gamma, cfg.vocab, dtype=torch.float32, device="cuda")
    gb.draft_batched(ids, anchors, tok, conf, lg)
    torch.cuda.synchronize()
    assert gb.check() == 0
    assert [gb.context_length(s) for s in (4, 1, 2, 0)] == [9, 0, 23, 0]
    dr = oracle.Drafter(cfg, W)
    for i, n in enumerate(lens):
        if n:
            dr.ingest(feats[i], seq=i)
    for i in range(3):
        check_block(dr, i, int(anchors[i]), tok[i].cpu().numpy(), conf[i].cpu().numpy(), lg[i].cpu().numpy(),
                    label=f"seq {i}")
    # cache placement of slot 4 (sequence 0) and slot 2 (sequence 2)
    for slot, i in ((4, 0), (2, 2)):
        for layer in range(cfg.n_layers):
            K, V = dr.cache(i, layer)
            gk, gv = gb.cache(slot, layer, lens[i])
            assert np.max(np.abs(tensor_to_f64(gk) - K)) <= 2e-2 * np.max(np.abs(K))
            assert np.max(np.abs(tensor_to_f64(gv) - V)) <= 2e-2 * np.max(np.abs(V))


def test_batched_many_sequences_ragged_vocab():
    """Eleven sequences (the many-sequence paths: gathered anchor embeddings and
    the Markov bias as one GEMM per position over all sequences), ragged
    context lengths including 0 and tile edges, V 1000 (not a multiple of the
    32-entry argmax chunks or the 128-row GEMM tiles), r 64, head_dim 64."""
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=128, n_heads=2, n_layers=2, ff_mult=2, gamma=4,
                            vocab=1000, markov_rank=64)
    W = syn.make_weights(cfg, seed=11, norm_std=0.1)
    lens = [0, 1, 5, 63, 64, 65, 130, 7, 200, 33, 90]
    n = len(lens)
    feats = [syn.make_feats(cfg, L, seed=11, seq=i) for i, L in enumerate(lens)]
    gb = make_gpu_drafter(cfg, weights_to_device(W), max_ctx=208, max_seqs=12)
    ids = torch.arange(n, dtype=torch.int32, device="cuda")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    gb.ingest_context_batched(ids, cu, to_torch(np.concatenate(feats, axis=0)))
    anchors = torch.tensor([0, 999, 31, 32, 500, 998, 1, 640, 2, 333, 768], dtype=torch.int32, device="cuda")
    tok = torch.empty(n, cfg.gamma, dtype=torch.int32, device="cuda")
    conf = torch.empty(n, cfg.gamma, dtype=torch.float32, device="cuda")
    lg = torch.empty(n, cfg.gamma, cfg.vocab, dtype=torch.float32, device="cuda")
    gb.draft_batched(ids, anchors, tok, conf, lg)
    torch.cuda.synchronize()
    assert gb.check() == 0
    dr = oracle.Drafter(cfg, W)
    for i, L in enumerate(lens):
        if L:
            dr.ingest(feats[i], seq=i)
    for i in range(n):
        check_block(dr, i, int(anchors[i]), tok[i].cpu().numpy(), conf[i].cpu().numpy(), lg[i].cpu().numpy(),
                    label=f"seq {i} (L {lens[i]})")


@pytest.mark.parametrize("n_heads,gamma,L", [(4, 5, 300), (8, 12, 50), (4, 8, 1500)])
def test_persistent_draft_layers(n_heads, gamma, L):
    """Every draft layer in one launch on warp MMAs (d and F multiples of 512,
    head dim 64 or 128): one or two 8-row block tiles, one key range (no merge)
    and many key ranges (merged), three draws in a row on the same handle."""
    import block_draft_model_gb300 as bdm
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=512, n_heads=n_heads, n_layers=2, ff_mult=2, gamma=gamma,
                            vocab=1000, markov_rank=32)
    dr, gdr, _ = _small(cfg, L, seed=15, chunks=[L // 2], anchors=[1, 998, 500], max_ctx=L + 16,
                        paths=[(bdm.PATH_LAYERS, bdm.LAYERS_PERSISTENT_MMA)])
    X = syn.make_feats(cfg, 3, seed=16)
    dr.ingest(X)
    gdr.ingest_context(to_torch(X))
    tok, conf, lg = _draft(gdr, cfg, 77)
    check_block(dr, 0, 77, tok, conf, lg, label="after 3 more rows")


# d, heads, gamma, L, vocab, hidden, layers, Markov rank
STEP_SHAPES = [
    (256, 2, 8, 300, 1000, 256, 2, 64),      # head_dim 128, one key range per head over 2 x 76 CTAs
    (128, 2, 16, 97, 777, 192, 2, 128),      # head_dim 64, all 16 block rows (both TMEM column groups), H % 64 != 0
    (384, 3, 5, 1500, 2053, 320, 3, 256),    # three heads of 128, many key ranges merged, ragged vocabulary tile
    (512, 8, 1, 40, 4096, 256, 1, 64),       # gamma 1 (no mask rows), eight heads of 64
    (256, 4, 7, 0, 1100, 256, 2, 32),        # empty context: the block attends to itself only; the separate chain
    (128, 2, 4, 50, 100, 128, 1, 64),        # fewer vocabulary rows than CTAs: CTAs without rows in the chain
]


@pytest.mark.parametrize("d,n_heads,gamma,L,vocab,hidden,n_layers,rank", STEP_SHAPES)
def test_one_launch_step_tc(d, n_heads, gamma, L, vocab, hidden, n_layers, rank):
    """The whole batch-1 step in one launch with tcgen05 projections: K blocks split over the
    CTAs with tiles shared by several CTAs (atomic reductions), key ranges of one head merged
    cooperatively, ragged weight tiles, and (rank 64 / 128 / 256) the Markov chain, argmax and
    confidences in the same launch; three draws in a row on the same handle, then more context
    and another draw."""
    import block_draft_model_gb300 as bdm
    cfg = syn.DrafterConfig(hidden=hidden, n_taps=2, d_draft=d, n_heads=n_heads, n_layers=n_layers, ff_mult=2,
                            gamma=gamma, vocab=vocab, markov_rank=rank)
    dr, gdr, _ = _small(cfg, L, seed=31, chunks=[L // 2] if L else [], anchors=[1, vocab - 1, vocab // 3],
                        max_ctx=L + 16, norm_std=0.3, paths=[(bdm.PATH_LAYERS, bdm.LAYERS_STEP_TC)])
    X = syn.make_feats(cfg, 3, seed=32)
    dr.ingest(X)
    gdr.ingest_context(to_torch(X))
    tok, conf, lg = _draft(gdr, cfg, 77 % vocab)
    check_block(dr, 0, 77 % vocab, tok, conf, lg, label="after 3 more rows")
    tok, conf, _ = _draft(gdr, cfg, 5, want_logits=False)  # without the logits output
    check_block(dr, 0, 5, tok, conf, None, label="no logits")
    assert gdr.check() == 0


@pytest.mark.parametrize("layers", ["per_kernel", "step_tc"])
def test_layer_forms_agree_without_graphs(layers):
    """The per-kernel and the one-launch forms, launched directly (no CUDA graph) with the
    anchor passed by value."""
    import block_draft_model_gb300 as bdm
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=256, n_heads=2, n_layers=2, ff_mult=2, gamma=6,
                            vocab=900, markov_rank=128)
    form = bdm.LAYERS_PER_KERNEL if layers == "per_kernel" else bdm.LAYERS_STEP_TC
    _small(cfg, 130, seed=33, chunks=[60], anchors=[3, 899, 450], norm_std=0.3,
           paths=[(bdm.PATH_GRAPHS, 1), (bdm.PATH_LAYERS, form)])


@pytest.mark.parametrize("gamma", [4, 16])
def test_separate_normalisation_launches(gamma):
    """Batch-1 layers one kernel per projection with a normalisation launch before each
    normalised projection; d 768 gives 12 K-blocks, the vocabulary a ragged last weight tile."""
    import block_draft_model_gb300 as bdm
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=768, n_heads=6, n_layers=2, ff_mult=2, gamma=gamma,
                            vocab=1100, markov_rank=32)
    _small(cfg, 200, seed=17, chunks=[90], anchors=[5, 1099], norm_std=0.3,
           paths=[(bdm.PATH_LAYERS, bdm.LAYERS_PER_KERNEL), (bdm.PATH_NORM_CHAIN, 1)])


@pytest.mark.parametrize("d,n_heads,gamma,L,vocab", [(512, 4, 8, 300, 1000), (64, 1, 16, 100, 777),
                                                     (768, 6, 5, 257, 1100)])
def test_norm_chain_through_residual_epilogues(d, n_heads, gamma, L, vocab):
    """Batch-1 layers without normalisation launches: the W_o and W_down
    epilogues write x, the next projection's operand bf16(x * g) and the
    8-column sums of x^2; QKV, gate/up and the vocabulary projection scale
    their accumulators by 1 / rms from those sums.  d 512 and 768 reduce
    split-K through clusters; d 64 runs W_o unsplit (the per-column epilogue);
    gamma 16 fills all 16 operand rows.  The per-kernel form is forced so the
    small shapes take it."""
    import block_draft_model_gb300 as bdm
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=d, n_heads=n_heads, n_layers=3, ff_mult=2, gamma=gamma,
                            vocab=vocab, markov_rank=32)
    dr, gdr, _ = _small(cfg, L, seed=18, chunks=[L // 3], anchors=[2, vocab - 1, vocab // 2], norm_std=0.3,
                        max_ctx=L + 8, paths=[(bdm.PATH_LAYERS, bdm.LAYERS_PER_KERNEL)])
    X = syn.make_feats(cfg, 2, seed=19)
    dr.ingest(X)
    gdr.ingest_context(to_torch(X))
    tok, conf, lg = _draft(gdr, cfg, 11)
    check_block(dr, 0, 11, tok, conf, lg, label="after 2 more rows")


def test_grouped_kv_more_tiles_than_sms():
    """Eq 3 K/V of 4 layers over 1280 new rows (d 512): 10 x 4 x 4 = 160 output tiles, more than one
    per SM, so the persistent CTAs take a second tile; every cache row is compared."""
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=512, n_heads=4, n_layers=4, ff_mult=2, gamma=4,
                            vocab=600, markov_rank=32)
    _small(cfg, 1280, seed=23, chunks=[], anchors=[9], max_ctx=1300)


def test_ingest_projection_split_over_k():
    """A context projection with few output tiles (300 rows, d 256) and a long
    K (4 taps x 512): the tensor-core GEMM cuts K into ranges whose partial
    products the normalisation sums."""
    cfg = syn.DrafterConfig(hidden=512, n_taps=4, d_draft=256, n_heads=2, n_layers=2, ff_mult=2, gamma=4,
                            vocab=600, markov_rank=32)
    _small(cfg, 300, seed=14, chunks=[], anchors=[3, 599])


@pytest.mark.parametrize("n_seq,rank,vocab,form", [
    (3, 64, 1000, "mma"), (1, 128, 5003, "mma"), (7, 256, 2048, "mma"),
    (3, 64, 1000, "fma"), (2, 128, 5003, "fma"), (1, 256, 73448, "fma"), (2, 256, 100003, "fma"),
    (1, 256, 150001, "fma"),
])
def test_markov_chain_few_sequences(n_seq, rank, vocab, form):
    """1 to 7 sequences with r in {64, 128, 256}: the whole Markov chain in one
    cooperative launch with the vocabulary slices resident on the SMs; the dot
    products on the tensor cores ("mma") or, for one or two sequences, on the
    FMA pipes with the argmax exchanged through per-CTA words ("fma").
    Vocabularies that leave ragged slices, CTAs without rows (V 1000), rows
    past the resident ones (V 73448) and several 512-row passes (V 100003);
    V 150001 with one sequence streams most of each slice through the
    per-thread copy ring (a ragged last block, a shorter last slice);
    three sequences then one on the same handle switch between the forms."""
    import block_draft_model_gb300 as bdm
    cfg = syn.DrafterConfig(hidden=128, n_taps=2, d_draft=128, n_heads=2, n_layers=1, ff_mult=2, gamma=6,
                            vocab=vocab, markov_rank=rank)
    W = syn.make_weights(cfg, seed=13, norm_std=0.1)
    lens = [17 + 5 * i for i in range(n_seq)]
    feats = [syn.make_feats(cfg, L, seed=13, seq=i) for i, L in enumerate(lens)]
    gb = make_gpu_drafter(cfg, weights_to_device(W), max_ctx=64, max_seqs=n_seq)
    if form == "mma":
        gb.set_path(bdm.PATH_MARKOV, 1)
    ids = torch.arange(n_seq, dtype=torch.int32, device="cuda")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    gb.ingest_context_batched(ids, cu, to_torch(np.concatenate(feats, axis=0)))
    anchors = torch.tensor([(37 * i + 5) % vocab for i in range(n_seq)], dtype=torch.int32, device="cuda")
    tok = torch.empty(n_seq, cfg.gamma, dtype=torch.int32, device="cuda")
    conf = torch.empty(n_seq, cfg.gamma, dtype=torch.float32, device="cuda")
    lg = torch.empty(n_seq, cfg.gamma, cfg.vocab, dtype=torch.float32, device="cuda")
    dr = oracle.Drafter(cfg, W)
    for i, L in enumerate(lens):
        dr.ingest(feats[i], seq=i)
    for rep in range(3):  # repeated launches alternate the argmax word sets
        gb.draft_batched(ids, anchors, tok, conf, lg)
        torch.cuda.synchronize()
        assert gb.check() == 0
        for i in range(n_seq):
            check_block(dr, i, int(anchors[i]), tok[i].cpu().numpy(), conf[i].cpu().numpy(), lg[i].cpu().numpy(),
                        label=f"launch {rep} seq {i}")
    if n_seq > 1:  # fewer sequences on the same handle: the other form's words and epoch stay consistent
        for rep in range(2):
            gb.draft_batched(ids[:1], anchors[:1], tok[:1], conf[:1], lg[:1])
            torch.cuda.synchronize()
            assert gb.check() == 0
            check_block(dr, 0, int(anchors[0]), tok[0].cpu().numpy(), conf[0].cpu().numpy(), lg[0].cpu().numpy(),
                        label=f"one sequence, launch {rep}")


# (context rows, capacity): the capacity bounds the keys the host plans the key ranges for, the
# actual length sizes them on the device.  Two heads: 16 ranges merged inside a thread-block cluster
# (707 and 1807 keys), 76 ranges with 8 of them filled (the one-pass merge by the last CTA) and 63 of
# them filled (the piecewise merge, several staged pieces).
ATTN_RANGES = [(700, 1900), (1800, 1900), (500, 8000), (7990, 8000)]


@pytest.mark.parametrize("ctx,cap", ATTN_RANGES)
def test_bf16_attention_many_key_ranges(ctx, cap):
    """head_dim 128, two heads: the keys of each head are split over many CTAs
    (64-key tiles, a ragged last tile) and merged, in each of the three forms."""
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=256, n_heads=2, n_layers=2, ff_mult=2, gamma=7,
                            vocab=1000, markov_rank=64)
    _small(cfg, ctx, seed=12, chunks=[700], anchors=[4, 998], max_ctx=cap)


def test_bf16_attention_long_ranges_head_dim_64():
    """head_dim 64, eight heads, about 10000 keys: one long range per SM (the deep cp.async ring),
    merged by the ticketed last CTA in staged pieces; gamma 8 fills the one 8-wide query tile."""
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=512, n_heads=8, n_layers=1, ff_mult=2, gamma=8,
                            vocab=1000, markov_rank=64)
    _small(cfg, 10000, seed=13, chunks=[4000], anchors=[3, 997], max_ctx=10100)


@pytest.mark.parametrize("ctx,cap", [(2000, 2100), (9000, 9100)])
def test_bf16_attention_partial_second_query_tile(ctx, cap):
    """gamma 11: the block queries fill one 8-wide tile and 3 rows of a second; four heads of 64.
    2000 keys: 16 short ranges merged inside a cluster; 9000 keys: 38 long ranges (one CTA per SM,
    the deep ring) merged by the ticketed last CTA in staged pieces."""
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=256, n_heads=4, n_layers=1, ff_mult=2, gamma=11,
                            vocab=1000, markov_rank=64)
    _small(cfg, ctx, seed=14, chunks=[ctx // 3], anchors=[7, 990], max_ctx=cap)


def test_host_checked_errors():
    import block_draft_model_gb300 as bdm
    cfg = syn.DrafterConfig(hidden=128, n_taps=2, d_draft=128, n_heads=2, n_layers=1, ff_mult=2, gamma=2,
                            vocab=300, markov_rank=8)
    W = syn.make_weights(cfg, seed=7)
    gdr = make_gpu_drafter(cfg, weights_to_device(W), max_ctx=10)
    X = to_torch(syn.make_feats(cfg, 11, seed=7))
    with pytest.raises(bdm.DsparkError) as e:
        gdr.ingest_context(X)
    assert e.value.status == bdm.ERR_CAPACITY
    assert gdr.context_length() == 0
    gdr.ingest_context(X[:10])
    assert gdr.context_length() == 10
    tok = torch.empty(2, dtype=torch.int32, device="cuda")
    conf = torch.empty(2, dtype=torch.float32, device="cuda")
    for bad in (-1, 300):
        with pytest.raises(bdm.DsparkError) as e:
            gdr.draft(bad, tok, conf)
        assert e.value.status == bdm.ERR_INVALID_ARG
    gdr.reset()
    assert gdr.context_length() == 0
    # device-side checks of the batched calls: a bad anchor and a bad slot set bits of the error word
    ids = torch.tensor([0], dtype=torch.int32, device="cuda")
    gdr.draft_batched(ids, torch.tensor([300], dtype=torch.int32, device="cuda"), tok.view(1, 2), conf.view(1, 2))
    assert gdr.check() & 1
    gdr.draft_batched(torch.tensor([3], dtype=torch.int32, device="cuda"),
                      torch.tensor([1], dtype=torch.int32, device="cuda"), tok.view(1, 2), conf.view(1, 2))
    assert gdr.check() & 2
    cu = torch.tensor([0, 11], dtype=torch.int32, device="cuda")
    gdr.ingest_context_batched(ids, cu, X)
    assert gdr.check() & 4
    assert gdr.context_length() == 0
    assert gdr.check() == 0


# --------------------------------------------------------------------------- full-size drafters

def test_minicpm_shaped_full_size():
    """MiniCPM-shaped drafter (H 2048, m 5, d 2048, 16 heads, 5 layers, gamma 8,
    V 73448, r 256), 1024 context rows, then draft; every cache row of sampled
    rows and every logit of two blocks are compared, for the default one-launch
    step and for the per-kernel form on a second handle."""
    import block_draft_model_gb300 as bdm
    wl = syn.WORKLOADS["minicpm_L1024"]
    cfg = wl.cfg
    W = syn.make_weights(cfg, seed=0)
    X = syn.make_feats(cfg, wl.ctx_len, seed=0)
    Wd = weights_to_device(W)
    anchors = syn.anchors(wl)[:, 0]
    outs = {}
    for form in (bdm.LAYERS_STEP_TC, bdm.LAYERS_PER_KERNEL):
        gdr = make_gpu_drafter(cfg, Wd, max_ctx=wl.ctx_len + 64)
        gdr.set_path(bdm.PATH_LAYERS, form)
        gdr.ingest_context(to_torch(X))
        outs[form] = [_draft(gdr, cfg, int(a)) for a in (anchors[0], 12345)]
        assert gdr.check() == 0
        if form == bdm.LAYERS_STEP_TC:
            keep = gdr
        else:
            gdr.close()
    dr = oracle.Drafter(cfg, W)
    dr.ingest(X)
    rows = np.unique(np.concatenate([[0, 1, 511, 1023], syn.uniform_int(9, 9, (28,), 0, 1023)]))
    check_cache(dr, keep, cfg, 0, rows, label="minicpm cache")
    for form, blocks in outs.items():
        for a, (tok, conf, lg) in zip((anchors[0], 12345), blocks):
            check_block(dr, 0, int(a), tok, conf, lg, label=f"minicpm form {form} anchor {a}")


@pytest.fixture(scope="module")
def gemma():
    cfg = syn.GEMMA
    W = syn.make_weights(cfg, seed=0)
    Wd = weights_to_device(W)
    dr = oracle.Drafter(cfg, W)
    return cfg, W, Wd, dr


def test_gemma_shaped_streaming_steps(gemma):
    """Gemma-shaped default DFlash (H 2560, m 4, d 1024, 8 heads, 5 layers,
    gamma 5, V 262144, r 256): 4096 context rows, then 64 steps that each ingest
    1-6 new rows and draft; steps 0, 1, 31 and 63 are checked."""
    cfg, W, Wd, dr = gemma
    wl = syn.WORKLOADS["gemma_L4096_stream"]
    anchors, counts = syn.anchors(wl)[:, 0], syn.step_counts(wl)[:, 0]
    total = wl.ctx_len + int(counts.sum())
    gdr = make_gpu_drafter(cfg, Wd, max_ctx=total + 8)
    X0 = syn.make_feats(cfg, wl.ctx_len, seed=0)
    gdr.ingest_context(to_torch(X0))
    dr.reset(0)
    dr.ingest(X0)
    check_at = {0, 1, 31, 63}
    for s in range(wl.steps):
        Xs = syn.make_feats(cfg, int(counts[s]), seed=0, step=s)
        gdr.ingest_context(to_torch(Xs))
        dr.ingest(Xs)
        want = s in check_at
        tok, conf, lg = _draft(gdr, cfg, int(anchors[s]), want_logits=want)
        if want:
            check_block(dr, 0, int(anchors[s]), tok, conf, lg, label=f"gemma step {s}")
    assert gdr.context_length() == total
    rows = np.array([0, 4095, 4096, total - 1])
    check_cache(dr, gdr, cfg, 0, rows, label="gemma cache")
    assert gdr.check() == 0
    dr.reset(0)


def test_gemma_shaped_long_context(gemma):
    """32768 context rows ingested at once, then 16 draft steps (0 and 15 checked)."""
    cfg, W, Wd, dr = gemma
    wl = syn.WORKLOADS["gemma_L32768_ingest"]
    X = syn.make_feats(cfg, wl.ctx_len, seed=0)
    gdr = make_gpu_drafter(cfg, Wd, max_ctx=wl.ctx_len)
    gdr.ingest_context(to_torch(X))
    anchors = syn.anchors(wl)[:, 0]
    outs = {}
    for s in range(wl.steps):
        o = _draft(gdr, cfg, int(anchors[s]), want_logits=s in (0, 15))
        if s in (0, 15):
            outs[s] = o
    assert gdr.check() == 0
    dr.reset(0)
    dr.ingest(X)
    rows = np.unique(np.concatenate([[0, 32767], syn.uniform_int(9, 10, (30,), 0, 32767)]))
    check_cache(dr, gdr, cfg, 0, rows, label="long cache")
    for s, (tok, conf, lg) in outs.items():
        check_block(dr, 0, int(anchors[s]), tok, conf, lg, label=f"long step {s}")
    dr.reset(0)


def test_gemma_shaped_batched_serving(gemma):
    """64 sequences with ragged contexts (512-8192 rows), 128 steps of 1-6 new
    rows per sequence and one block per sequence.  Four sequences are checked
    with every logit at steps 0 and 127, and the tokens and confidences of all
    64 sequences at step 0 (the oracle re-ingests one sequence at a time)."""
    cfg, W, Wd, dr = gemma
    wl = syn.WORKLOADS["gemma_batched64"]
    n = wl.n_seqs
    lens = syn.ctx_lengths(wl)
    counts = syn.step_counts(wl)
    anchors = syn.anchors(wl)
    max_ctx = int(lens.max() + counts.sum(axis=0).max()) + 8
    gdr = make_gpu_drafter(cfg, Wd, max_ctx=max_ctx, max_seqs=n)
    ids = torch.arange(n, dtype=torch.int32, device="cuda")

    def ingest(step, cnts):
        feats = [syn.make_feats(cfg, int(c), seed=0, step=step, seq=i) for i, c in enumerate(cnts)]
        cu = torch.tensor(np.concatenate([[0], np.cumsum(cnts)]), dtype=torch.int32, device="cuda")
        gdr.ingest_context_batched(ids, cu, to_torch(np.concatenate(feats, axis=0)))
        return feats

    first = ingest(-1, lens)
    sample = [0, 17, int(np.argmax(lens)), int(np.argmin(lens))]
    kept = {i: [first[i]] for i in sample}
    del first
    tok = torch.empty(n, cfg.gamma, dtype=torch.int32, device="cuda")
    conf = torch.empty(n, cfg.gamma, dtype=torch.float32, device="cuda")
    lg = torch.empty(n, cfg.gamma, cfg.vocab, dtype=torch.float32, device="cuda")
    results = {}
    for s in range(wl.steps):
        feats = ingest(s, counts[s])
        for i in sample:
            kept[i].append(feats[i])
        want = s in (0, wl.steps - 1)
        gdr.draft_batched(ids, to_torch(anchors[s]), tok, conf, lg if want else None)
        if want:
            torch.cuda.synchronize()
            results[s] = {i: (tok[i].cpu().numpy(), conf[i].cpu().numpy(), lg[i].cpu().numpy(),
                              len(kept[i])) for i in sample}
            if s == 0:
                first_tok, first_conf = tok.cpu().numpy().copy(), conf.cpu().numpy().copy()
    assert gdr.check() == 0
    for i in sample:
        assert gdr.context_length(i) == int(lens[i] + counts[:, i].sum())
    for s, per in results.items():
        for i, (t, c, l, nparts) in per.items():
            dr.reset(0)
            for part in kept[i][:nparts]:
                dr.ingest(part)
            check_block(dr, 0, int(anchors[s, i]), t, c, l, label=f"batched step {s} seq {i}")
    # the whole batch at step 0: every sequence's block must be one of the oracle's valid chains
    for i in range(n):
        dr.reset(0)
        dr.ingest(syn.make_feats(cfg, int(lens[i]), seed=0, step=-1, seq=i))
        dr.ingest(syn.make_feats(cfg, int(counts[0, i]), seed=0, step=0, seq=i))
        check_block(dr, 0, int(anchors[0, i]), first_tok[i], first_conf[i], None, label=f"batched step 0 seq {i}")
    dr.reset(0)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_ingest_and_draft_matches_two_calls(dtype):
    """dspark_ingest_and_draft = dspark_ingest_context then dspark_draft: the same tokens, confidences
    and logits, bit for bit (its block rows, and for bf16 layer 0's QKV projection, run on a side
    stream while the rows are ingested), over several steps: long ingests (tile GEMMs), short ones
    (weight-streaming or SIMT GEMMs, beside the side stream's own split-K launches) and one with no
    new rows."""
    import block_draft_model_gb300 as bdm
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=256, n_heads=2, n_layers=2, ff_mult=2, gamma=6,
                            vocab=1000, markov_rank=64, dtype=dtype)
    W = syn.make_weights(cfg, seed=21)
    Wd = weights_to_device(W)
    feats = to_torch(syn.make_feats(cfg, 300, seed=21))
    a = make_gpu_drafter(cfg, Wd, max_ctx=400)
    b = make_gpu_drafter(cfg, Wd, max_ctx=400)
    for g in (a, b):  # launched directly: the graphed draft plans its key ranges for the capacity, not the length
        g.set_path(bdm.PATH_GRAPHS, 1)
    for lo, hi, anchor in [(0, 200, 5), (200, 250, 17), (250, 250, 999), (250, 255, 3), (255, 256, 640),
                           (256, 300, 8)]:
        ta = torch.empty(cfg.gamma, dtype=torch.int32, device="cuda")
        tb = torch.empty_like(ta)
        ca = torch.empty(cfg.gamma, dtype=torch.float32, device="cuda")
        cb = torch.empty_like(ca)
        la = torch.empty(cfg.gamma, cfg.vocab, dtype=torch.float32, device="cuda")
        lb = torch.empty_like(la)
        if hi > lo:
            a.ingest_context(feats[lo:hi])
        a.draft(anchor, ta, ca, la)
        b.ingest_and_draft(feats[lo:hi], anchor, tb, cb, lb)
        torch.cuda.synchronize()
        assert torch.equal(ta, tb), (lo, hi)
        assert torch.equal(ca, cb), (lo, hi)
        assert torch.equal(la, lb), (lo, hi)
        assert a.context_length() == b.context_length() == hi
    assert a.check() == 0 and b.check() == 0

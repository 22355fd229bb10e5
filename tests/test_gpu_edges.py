"""Edge cases of the CUDA path against the oracle: padding (V < K), ties, -inf,
misaligned rows and base pointers, rows split over many CTAs, device-side errors."""

import numpy as np
import pytest
import torch

import ragged_log_probs_gb300 as lp
import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    parity.ensure_built()


def _custom(logits, lengths, echo, levels, seed=0, **kw):
    return workloads.make_custom_batch(logits.cuda().contiguous(), lengths, echo, levels, seed=seed, **kw)


@pytest.mark.parametrize("V", [1, 2, 3, 5, 7, 9])
@pytest.mark.parametrize("levels", [3, 6])
def test_vocab_smaller_than_k_pads(V, levels):
    g = torch.Generator().manual_seed(V)
    x = torch.randn(6, V, generator=g) * 2
    b = _custom(x, [2, 3, 1], [1, 0, 1], levels, seed=V)
    parity.check_batch(b)
    _, _, tok = parity.run_gpu(b)
    K = 2 ** levels - 1
    if V < K:
        assert np.all(tok[:, V:K] == 0xFFFFFFFF)


def test_all_equal_rows():
    x = torch.full((5, 3001), 0.75)
    b = _custom(x, [5], [1], 6)
    parity.check_batch(b)
    _, out_lp, tok = parity.run_gpu(b)
    assert tok[:, :63].tolist() == [list(range(63))] * 5
    np.testing.assert_allclose(out_lp, -np.log(3001), atol=1e-5)


def test_quantised_ties_everywhere():
    g = torch.Generator().manual_seed(3)
    x = torch.round(torch.randn(40, 20000, generator=g) * 4) / 4
    b = _custom(x, [10, 30], [1, 1], 6)
    parity.check_batch(b)


def test_neg_inf_rows():
    g = torch.Generator().manual_seed(4)
    x = torch.randn(6, 1000, generator=g)
    x[0, :] = float("-inf")                      # all -inf: NaN logprobs, ids by order rule
    x[1, 3:] = float("-inf")                      # fewer finite entries than K
    x[2, ::2] = float("-inf")
    x[3, 500] = 40.0                              # one dominant entry
    b = _custom(x, [6], [1], 3)
    parity.check_batch(b)


@pytest.mark.parametrize("V", [4093, 4094, 4095, 4097, 32001])
def test_odd_vocab_misaligned_rows(V):
    g = torch.Generator().manual_seed(V)
    x = torch.randn(9, V, generator=g) * 2
    b = _custom(x, [4, 1, 4], [1, 0, 1], 3)
    parity.check_batch(b)


@pytest.mark.parametrize("shift", [1, 2, 3])
def test_misaligned_base_pointer(shift):
    T, V = 7, 8000
    g = torch.Generator().manual_seed(shift)
    flat = torch.empty(T * V + 4, device="cuda")
    x = flat[shift:shift + T * V].view(T, V)
    x.copy_((torch.randn(T, V, generator=g) * 2).cuda())
    assert x.data_ptr() % 16 != 0
    b = workloads.make_custom_batch(x, [3, 4], [1, 1], 3, seed=shift)
    parity.check_batch(b)


@pytest.mark.parametrize("B,V,levels", [(1, 256000, 6), (1, 128256, 3), (3, 152064, 3), (2, 1000003, 3),
                                        (1, 5000, 0), (5, 777777, 6)])
def test_rows_split_over_many_ctas(B, V, levels):
    b = workloads.make_next_token_batch(B, V, levels=levels, dist="normal", scale=3.0, device="cuda", seed=V)
    parity.check_batch(b)


def test_split_path_repeatable_counters_reset():
    b = workloads.make_next_token_batch(3, 200000, levels=3, device="cuda", seed=9)
    ws = lp.new_workspace(b.B, b.T, b.V, b.levels)
    first = parity.run_gpu(b, workspace=ws)
    for _ in range(3):
        again = parity.run_gpu(b, workspace=ws)
        for x, y in zip(first, again):
            assert np.array_equal(x, y, equal_nan=True) if x.dtype.kind == "f" else np.array_equal(x, y)


def test_single_token_sequences_and_b1():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(1, 777, generator=g)
    parity.check_batch(_custom(x, [1], [1], 3))
    parity.check_batch(_custom(x, [1], [0], 3))
    x = torch.randn(4, 777, generator=g)
    parity.check_batch(_custom(x, [1, 1, 1, 1], [1, 0, 1, 0], 2))


def test_many_batches_global_offsets_path():
    # B+1 above the shared-memory staging limit: offsets are read from global memory.
    B = 3000
    g = torch.Generator().manual_seed(6)
    x = torch.randn(B + 100, 64, generator=g)
    lengths = [1] * (B - 1) + [101]
    echo = [i % 3 == 0 for i in range(B)]
    parity.check_batch(_custom(x, lengths, echo, 3))


def test_token_out_of_range_sets_status_and_nan():
    g = torch.Generator().manual_seed(7)
    x = torch.randn(4, 300, generator=g)
    b = _custom(x, [4], [1], 3, tokens=[1, 2, 300, 3], sampled=[5])
    ws = lp.new_workspace(b.B, b.T, b.V, b.levels)
    out_off = lp.plan(b.logit_row_offsets, b.echo, b.T, ws)
    out_lp = torch.empty((4, 8), device="cuda")
    out_tok = torch.empty((4, 8), dtype=torch.int32, device="cuda")
    lp.compute(b.logits, b.logit_row_offsets, b.tokens, b.sampled_tokens, out_off, b.echo, 3, out_lp, out_tok, ws)
    status = lp.read_status(ws)
    assert status == (1 << 5)
    olp = out_lp.cpu().numpy()
    otok = out_tok.cpu().numpy().view(np.uint32)
    assert np.isnan(olp[1, 7]) and otok[1, 7] == 300          # row 1 scores token index 2 (= 300)
    assert not np.isnan(olp[0, 7]) and not np.isnan(olp[2, 7])
    ref = parity.oracle_for(b)
    assert not ref[3]
    parity.compare(olp, otok.astype(np.uint64), ref[1], ref[2], "token range")


def test_bad_offsets_detected_on_device():
    x = torch.randn(6, 100).cuda()
    off = torch.tensor([0, 3, 3, 6], dtype=torch.int32, device="cuda")   # empty batch 1
    echo = torch.ones(3, dtype=torch.uint8, device="cuda")
    ws = lp.new_workspace(3, 6, 100, 3)
    host = torch.zeros(2, dtype=torch.int32).pin_memory()
    lp.plan(off, echo, 6, ws, host_out=host)
    torch.cuda.synchronize()
    assert int(host[1]) == (1 << 4)
    off2 = torch.tensor([0, 3, 7], dtype=torch.int32, device="cuda")      # past T
    lp.plan(off2, echo[:2], 6, ws, host_out=host)
    torch.cuda.synchronize()
    assert int(host[1]) == (1 << 4)
    with pytest.raises(lp.LpError):
        lp.ragged_log_probs(x, off, torch.zeros(6, dtype=torch.int32, device="cuda"),
                            torch.zeros(3, dtype=torch.int32, device="cuda"), echo, 3)


@pytest.mark.parametrize("kernel", ["warp", "queue"])
@pytest.mark.parametrize("name,kw", [("decode", dict(B=40)), ("prefill", dict(B=3, max_len=90)),
                                     ("mixed", dict(B=9, max_len=20)), ("wide", dict(B=2, max_len=12)),
                                     ("tiny", dict())])
def test_both_kernels(kernel, name, kw, monkeypatch):
    # Warp-owned ranges and the CTA row queue must give the same result on every shape.
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    parity.check_batch(workloads.make_batch(name, "cuda", **kw), what=f"{name}/{kernel}")


@pytest.mark.parametrize("kernel", ["warp", "queue"])
def test_both_kernels_edge_rows(kernel, monkeypatch):
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    g = torch.Generator().manual_seed(11)
    x = torch.randn(7, 4097, generator=g)
    x[2, :] = float("-inf")
    x[4, 7:] = float("-inf")
    parity.check_batch(_custom(x, [2, 5], [1, 1], 6), what=f"edge/{kernel}")
    b = workloads.make_next_token_batch(3, 200003, levels=3, device="cuda", seed=12)
    ws = lp.new_workspace(b.B, b.T, b.V, b.levels)
    first = parity.run_gpu(b, workspace=ws)
    again = parity.run_gpu(b, workspace=ws)      # queue words and tickets were reset
    assert np.array_equal(first[2], again[2]) and np.array_equal(first[1], again[1], equal_nan=True)


@pytest.mark.parametrize("kernel", ["warp", "queue"])
@pytest.mark.parametrize("levels", [1, 2, 3])
def test_top_elements_in_one_lane(kernel, levels, monkeypatch):
    # Rows whose top-k sits in few lanes' elements or is decided by ties: all-equal rows,
    # coarse ties, top values planted in one lane's vectors, a row of few finite values.
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    g = torch.Generator().manual_seed(20 + levels)
    V = 40000
    x = torch.randn(8, V, generator=g)
    x[0, :] = 1.5
    x[1] = torch.round(x[1] * 2) / 2
    for j, pos in enumerate([0, 1, 2, 3, 128, 129, 130, 131]):
        x[2, pos] = 10.0 - 0.25 * j
    for j in range(8):
        x[3, 4 * 7 + 512 * j] = 9.0 + j
    x[4, :] = float("-inf")
    x[4, 5:12] = 2.0
    b = _custom(x, [3, 5], [1, 1], levels, seed=levels)
    parity.check_batch(b, what=f"one-lane/{kernel}/levels{levels}")


@pytest.mark.parametrize("V", [4093, 40001])
def test_top_elements_in_one_lane_misaligned(V):
    g = torch.Generator().manual_seed(V)
    x = torch.randn(6, V, generator=g)
    x[1, :] = 0.25
    x[2, 1:9] = 50.0
    parity.check_batch(_custom(x, [6], [1], 3, seed=V), what=f"one-lane-misaligned/{V}")


@pytest.mark.parametrize("kernel", ["warp", "queue"])
def test_compute_twice_after_one_plan(kernel, monkeypatch):
    # The row kernels leave their queue and ticket words cleared, so a second compute on
    # the same plan (no plan in between) gives the same rows, bit for bit (both kernels
    # split rows statically: the summation order does not depend on timing).
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    b = workloads.make_next_token_batch(40, 150001, levels=3, device="cuda", seed=21)
    ws = lp.new_workspace(b.B, b.T, b.V, b.levels)
    out_off = lp.plan(b.logit_row_offsets, b.echo, b.T, ws)
    outs = []
    for _ in range(3):
        o_lp = torch.empty((b.B, 8), device="cuda")
        o_tok = torch.empty((b.B, 8), dtype=torch.int32, device="cuda")
        lp.compute(b.logits, b.logit_row_offsets, b.tokens, b.sampled_tokens, out_off, b.echo, 3, o_lp, o_tok, ws)
        assert lp.read_status(ws) == 0
        outs.append((o_lp.cpu().numpy(), o_tok.cpu().numpy()))
    for lp_, tok_ in outs[1:]:
        assert np.array_equal(tok_, outs[0][1]) and np.array_equal(lp_, outs[0][0])
    ref = parity.oracle_for(b)
    parity.compare(outs[0][0], outs[0][1].view(np.uint32).astype(np.uint64), ref[1], ref[2], "twice")


@pytest.mark.parametrize("split", [1, 2, 7, 64])
@pytest.mark.parametrize("B,V,levels", [(1, 128256, 3), (5, 20011, 6), (13, 111, 3), (40, 50000, 0), (3, 9999, 1)])
def test_split_vocab_pieces(split, B, V, levels, monkeypatch):
    # Row-queue kernel with each row cut into `split` pieces (more pieces than vectors
    # leaves some empty), merged by the CTA that takes the row's last ticket.
    monkeypatch.setenv("LP_RAGGED_KERNEL", "queue")
    monkeypatch.setenv("LP_RAGGED_SPLIT", str(split))
    b = workloads.make_next_token_batch(B, V, levels=levels, dist="normal", scale=3.0, device="cuda",
                                        seed=B * 31 + split)
    parity.check_batch(b, what=f"split={split} B={B} V={V} levels={levels}")


@pytest.mark.parametrize("split", [3, 17])
def test_split_vocab_pieces_echo_and_variants(split, monkeypatch):
    monkeypatch.setenv("LP_RAGGED_KERNEL", "queue")
    monkeypatch.setenv("LP_RAGGED_SPLIT", str(split))
    b = workloads.make_batch("mixed", "cuda", B=6, max_len=9, V=30011, seed=90 + split)
    parity.check_batch(b, what=f"mixed split={split}")
    bv = workloads.with_temperatures(workloads.make_batch("mixed", "cuda", B=6, max_len=9, V=30011,
                                                          variable_extra=2, seed=91), seed=split)
    parity.check_batch(bv, what=f"variable+tau split={split}")


@pytest.mark.parametrize("B,V,levels,per_sm", [
    (151, 20000, 3, None), (152, 20000, 3, None), (153, 20000, 3, None), (304, 20000, 3, None),
    (305, 20000, 3, None), (456, 8000, 3, 3), (457, 8000, 3, 3), (456, 70000, 3, 3), (457, 70000, 3, 3),
    (1064, 16000, 3, 7), (1065, 16000, 3, 7), (1065, 100000, 3, 7), (1065, 100000, 6, 7)])
def test_kernel_choice_boundary(B, V, levels, per_sm):
    # The library's own choice: split pieces below one row per SM, whole rows up to three
    # per SM; then the row queue up to seven rows per SM for rows of 60 KB or more, for any
    # count of rows of 384 KB or more at K <= 31, else warp ranges. per_sm: the boundary
    # the case sits at (on 152 SMs); the expected kernel follows the rule on this GPU.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    row_bytes = 4 * V
    want = ("queue" if B <= 3 * sms or (row_bytes >= 60 * 1024 and B <= 7 * sms)
            or (1 <= levels <= 5 and row_bytes >= 384 * 1024) else "warp")
    assert lp.row_kernel(B, B, V, levels) == want
    b = workloads.make_next_token_batch(B, V, levels=levels, dist="normal", scale=3.0, device="cuda", seed=B)
    parity.check_batch(b, rows=parity.sample_rows(B, 40, seed=B), what=f"B={B} V={V} levels={levels} ({want})")


@pytest.mark.parametrize("kernel", ["warp", "queue"])
@pytest.mark.parametrize("quantised", [False, True])
def test_levels5_long_rows(kernel, quantised, monkeypatch):
    # top-31 over long rows: the row queue bounds it by the 16th largest of each lane
    # position's second-best lane maximum across its warps; quantised logits put many
    # elements exactly on that bound.
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    g = torch.Generator().manual_seed(55)
    x = torch.randn(24, 128256, generator=g) * 3
    if quantised:
        x = torch.round(x * 2) / 2
    b = workloads.make_custom_batch(x.cuda(), [1] * 24, [0] * 24, 5, seed=55)
    parity.check_batch(b, what=f"levels 5/{kernel}/{'quantised' if quantised else 'normal'}")


@pytest.mark.parametrize("kernel", ["warp", "queue"])
@pytest.mark.parametrize("B", [1025, 2047])
def test_many_batches_staged_row_lookup(kernel, B, monkeypatch):
    # Up to 2047 batches the offsets sit in shared memory and a row's batch is found with two
    # ballot rounds (at B = 2047 each lane's stride is 64 entries: two rounds of 32 lanes).
    # Uneven echo counts make the output offsets jump unevenly.
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    rng = np.random.default_rng(B)
    lengths = rng.integers(1, 4, size=B)
    echo = (rng.random(B) < 0.5).astype(np.int64)
    g = torch.Generator().manual_seed(B)
    x = torch.randn(int(lengths.sum()), 257, generator=g).cuda()
    b = _custom(x, lengths.tolist(), echo.tolist(), 3, seed=B)
    parity.check_batch(b, what=f"B={B}/{kernel}")


def test_decode_full_size_levels6_sampled():
    b = workloads.make_batch("decode", "cuda", levels=6)
    parity.check_batch(b, rows=parity.sample_rows(b.B, 16, seed=6), what="decode levels 6")


@pytest.mark.parametrize("kernel", ["warp", "queue"])
def test_levels6_quantised_ties(kernel, monkeypatch):
    # The top-63 bound compares with >= against a real element's value: elements equal to
    # it must still reach the candidates (many exact ties).
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    g = torch.Generator().manual_seed(14)
    x = (torch.round(torch.randn(9, 40000, generator=g) * 4) / 4).cuda()
    b = workloads.make_custom_batch(x, [1] * 9, [0] * 9, 6, seed=14)
    parity.check_batch(b, what=f"levels 6 ties/{kernel}")


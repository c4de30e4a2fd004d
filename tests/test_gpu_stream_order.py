"""Stream order across back-to-back launches (every kernel of the library is launched as a
programmatic dependent and waits for the kernel before it before touching global memory): a torch
kernel that writes the ids right before the fused call, the hash call feeding the lookup, the gate
consuming its own output, also inside a CUDA graph; each against an unpipelined run or the oracle
(GPU only)."""
import numpy as np
import pytest
import torch

import gram_hash_embedding_gb300 as geng
import synth
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    H.build_all()
    wl = synth.make_workload(0, full64=True)
    Ws, Ss = H.device_tables(wl)
    yield wl, Ws, Ss


def test_producer_kernel_then_fused_call(tiny):
    wl, Ws, Ss = tiny
    lay = wl.layout
    rng = np.random.default_rng(91)
    B, L, steps = 4, 48, 24
    srcs = [H.to_dev(rng.integers(0, lay.raw_vocab, size=(B, L))) for _ in range(steps)]
    ids = torch.empty((B, L), dtype=torch.int64, device="cuda")
    out = [torch.empty((B, L, lay.n_cols, lay.head_dim), dtype=torch.bfloat16, device="cuda")]
    hashes = torch.empty((B, L, 1, lay.n_cols), dtype=torch.int64, device="cuda")
    st, orc = H.make_state(wl, B, L * steps), H.make_oracle(wl, B, L * steps)
    kept_h, kept_r = [], []
    for k in range(steps):  # no synchronisation anywhere in the loop
        torch.add(srcs[k], 0, out=ids)  # a torch kernel writes the ids the next launch reads
        st.hash_lookup(ids, Ws, Ss, start_pos=k * L, out=out, hashes=hashes)
        kept_h.append(hashes.clone())
        kept_r.append(out[0].clone())
    torch.cuda.synchronize()
    for k in range(steps):
        exp_h, _ = orc.hash(srcs[k].cpu().numpy(), k * L)
        H.assert_bits_equal(kept_h[k].cpu().numpy(), exp_h, f"step {k} hashes")
        H.assert_bits_equal(H.bf16_bits(kept_r[k]), H.oracle_lookup_rows(wl, 0, exp_h[:, :, 0, :]), f"step {k} rows")


def test_hash_then_lookup_and_graph_replay(tiny):
    wl, Ws, Ss = tiny
    lay = wl.layout
    rng = np.random.default_rng(92)
    B, L = 3, 40
    ids = H.to_dev(rng.integers(0, lay.raw_vocab, size=(B, L)))
    fused_state, split_state = H.make_state(wl, B, 4096), H.make_state(wl, B, 4096)
    hashes = torch.empty((B, L, 1, lay.n_cols), dtype=torch.int64, device="cuda")
    rows = torch.empty((B * L * lay.n_cols, lay.head_dim), dtype=torch.bfloat16, device="cuda")
    fused = [torch.empty((B, L, lay.n_cols, lay.head_dim), dtype=torch.bfloat16, device="cuda")]
    sp = torch.zeros(B, dtype=torch.int32, device="cuda")

    def step():  # the lookup reads what the hash call just wrote; the start advances on the device
        split_state.hash(ids, sp, hashes=hashes)
        split_state.lookup(hashes.view(-1), Ws[0], Ss[0], out=rows)
        fused_state.hash_lookup(ids, Ws, Ss, start_pos=sp, out=fused)
        torch.add(sp, L, out=sp)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    assert torch.equal(rows.view(torch.int16), fused[0].reshape(-1, lay.head_dim).view(torch.int16))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(20):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(rows.view(torch.int16), fused[0].reshape(-1, lay.head_dim).view(torch.int16))
    assert int(sp[0]) == L * (3 + 20)  # capture records the step without running it
    assert fused_state.status() == 0 and split_state.status() == 0


def test_gate_consumes_its_own_output():
    H.build_all()
    torch.manual_seed(93)
    T, hc, dim = 512, 4, 256
    x = torch.randn((T, hc, dim)).to(torch.bfloat16).cuda()
    kv = torch.randn((T, (hc + 1) * dim)).to(torch.bfloat16).cuda()
    qw = torch.rand((hc, dim)).add_(0.5).to(torch.bfloat16).cuda()
    kw = torch.rand((hc, dim)).add_(0.5).to(torch.bfloat16).cuda()
    ref = x.clone()
    for _ in range(6):  # one launch at a time, synchronised
        ref = geng.engram_gate(ref, kv, qw, kw)
        torch.cuda.synchronize()
    y = x.clone()
    for _ in range(6):  # back to back, in place: each launch reads what the previous one wrote
        geng.engram_gate(y, kv, qw, kw, out=y)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


def test_l2_fetch_granularity_changes_no_result(tiny):
    """The context's L2 fetch granularity limit is a cache policy: hash ids and rows are the same
    at 32 bytes as at the context default, and the previous value comes back for the restore."""
    wl, Ws, Ss = tiny
    lay = wl.layout
    ids = H.to_dev(np.random.default_rng(94).integers(0, lay.raw_vocab, size=(2, 64)))
    st_a, st_b = H.make_state(wl, 2, 64), H.make_state(wl, 2, 64)
    ref = st_a.hash_lookup(ids, Ws, Ss)
    default = geng.set_l2_fetch_granularity(32)
    try:
        assert default in (0, 32, 64, 128)
        got = st_b.hash_lookup(ids, Ws, Ss)
        torch.cuda.synchronize()
        for r, g in zip(ref, got):
            assert torch.equal(r.view(torch.int16), g.view(torch.int16))
        assert geng.set_l2_fetch_granularity(default) == 32
    finally:
        geng.set_l2_fetch_granularity(default)
    with pytest.raises(geng.EngramError):
        geng.set_l2_fetch_granularity(48)


def test_explicit_side_stream_with_wrapper_temporaries(tiny):
    """A call on a stream other than the current one, with an int start_pos and outputs left to the
    wrapper: the start_pos array and the outputs are made on the current stream, so the named stream
    must wait for it and keep them alive until its kernel is done. Each step first makes garbage on
    the current stream (allocations that would reuse freed blocks), then calls on the side stream;
    every step's results must equal the oracle's."""
    wl, Ws, Ss = tiny
    lay = wl.layout
    rng = np.random.default_rng(17)
    B, L, steps = 2, 40, 12
    st, orc = H.make_state(wl, B, L * steps), H.make_oracle(wl, B, L * steps)
    side = torch.cuda.Stream()
    got_h, got_r, host_ids = [], [], []
    for k in range(steps):
        ids_h = rng.integers(0, lay.raw_vocab, size=(B, L))
        host_ids.append(ids_h)
        ids = H.to_dev(ids_h)
        torch.cuda.current_stream().wait_stream(side)  # ids reuse memory the side stream may still read
        junk = torch.full((1 << 16,), 7, dtype=torch.int32, device="cuda")  # current-stream traffic
        del junk
        hashes = geng.engram_hash(st.handle, ids, k * L, stream=side)
        with torch.cuda.stream(side):
            idx = hashes[:, :, 0, :].contiguous()
        rows = geng.engram_lookup(idx, Ws[0], Ss[0], lay.block, stream=side)
        with torch.cuda.stream(side):
            got_h.append(hashes.clone())
            got_r.append(rows.clone())
            ids.record_stream(side)
    torch.cuda.synchronize()
    for k in range(steps):
        exp_h, _ = orc.hash(host_ids[k], k * L)
        H.assert_bits_equal(got_h[k].cpu().numpy(), exp_h, f"side-stream hashes, step {k}")
        H.assert_bits_equal(H.bf16_bits(got_r[k]), H.oracle_lookup_rows(wl, 0, exp_h[:, :, 0, :]),
                            f"side-stream rows, step {k}")
    assert st.status() == 0


def test_fused_call_whose_ids_the_previous_launch_wrote(tiny):
    """A fused call may read its inputs before the kernel ahead of it completes only when this
    library's previous launch on the stream does not write them. Here it does: call 1 writes its
    int64 hash ids into H, and call 2, enqueued right behind it with nothing in between, takes H as its
    token ids (values up to ~9,000 against a vocabulary of 1,000: most are flagged and treated as
    masked, the rest map through token_map). H starts as -5 everywhere, so a call 2 that read H early
    would see -5 ids and hash masked tokens instead. Repeated, with fresh sentinels, in both orders
    of a large and a small call."""
    wl, Ws, Ss = tiny
    lay = wl.layout
    rng = np.random.default_rng(23)
    for B, L in ((4, 2048), (2, 96)):
        C = lay.n_cols
        st1, orc1 = H.make_state(wl, B, L), H.make_oracle(wl, B, L)
        st2, orc2 = H.make_state(wl, B, L * C), H.make_oracle(wl, B, L * C)
        ids1 = rng.integers(0, lay.raw_vocab, size=(B, L))
        hbuf = torch.full((B, L, 1, C), -5, dtype=torch.int64, device="cuda")
        out1 = [torch.empty((B, L, C, lay.head_dim), dtype=torch.bfloat16, device="cuda")]
        out2 = [torch.empty((B, L * C, C, lay.head_dim), dtype=torch.bfloat16, device="cuda")]
        h2 = torch.empty((B, L * C, 1, C), dtype=torch.int64, device="cuda")
        ids1_d = H.to_dev(ids1)
        torch.cuda.synchronize()
        st1.hash_lookup(ids1_d, Ws, Ss, start_pos=0, out=out1, hashes=hbuf)
        st2.hash_lookup(hbuf.view(B, L * C), Ws, Ss, start_pos=0, out=out2, hashes=h2)
        torch.cuda.synchronize()
        exp1, _ = orc1.hash(ids1, 0)
        H.assert_bits_equal(hbuf.cpu().numpy(), exp1, "call 1 hash ids")
        exp2, _ = orc2.hash(exp1.reshape(B, L * C), 0)
        H.assert_bits_equal(h2.cpu().numpy(), exp2, "call 2 hash ids (its ids are call 1's output)")
        H.assert_bits_equal(H.bf16_bits(out2[0]), H.oracle_lookup_rows(wl, 0, exp2[:, :, 0, :]), "call 2 rows")
        st1.status()
        st2.status()


def test_packed_call_whose_ids_the_previous_launch_wrote(tiny):
    """The same for a packed (continuous batching) call: call 1 writes its int64 hash ids into H, and
    a packed call enqueued right behind it takes H, flattened, as the token ids of sequences of ragged
    lengths (one of them empty), each at start position 0, so most of its tiles are past the cache
    halo. Packed calls read nothing before the kernel ahead of them completes; H starts as -5
    everywhere, so a call that did would hash masked tokens instead."""
    wl, Ws, Ss = tiny
    lay = wl.layout
    rng = np.random.default_rng(29)
    C = lay.n_cols
    B1, L1 = 2, 512
    lens = np.array([700, 0, 13, 300, 1], dtype=np.int64)
    T = int(lens.sum())
    assert T <= B1 * L1 * C
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    B2 = lens.size
    st1, orc1 = H.make_state(wl, B1, L1), H.make_oracle(wl, B1, L1)
    st2, orc2 = H.make_state(wl, B2, int(lens.max())), H.make_oracle(wl, B2, int(lens.max()))
    ids1 = rng.integers(0, lay.raw_vocab, size=(B1, L1))
    hbuf = torch.full((B1, L1, 1, C), -5, dtype=torch.int64, device="cuda")
    out1 = [torch.empty((B1, L1, C, lay.head_dim), dtype=torch.bfloat16, device="cuda")]
    h2 = torch.empty((T, 1, C), dtype=torch.int64, device="cuda")
    out2 = [torch.empty((T, C, lay.head_dim), dtype=torch.bfloat16, device="cuda")]
    cu_d, starts_d = H.to_dev(cu), H.to_dev(np.zeros(B2, dtype=np.int32))
    torch.cuda.synchronize()
    st1.hash_lookup(H.to_dev(ids1), Ws, Ss, start_pos=0, out=out1, hashes=hbuf)
    st2.hash_lookup_varlen(hbuf.view(-1)[:T], cu_d, starts_d, Ws, Ss, out=out2, hashes=h2, max_len=int(lens.max()))
    torch.cuda.synchronize()
    exp1, _ = orc1.hash(ids1, 0)
    H.assert_bits_equal(hbuf.cpu().numpy(), exp1, "call 1 hash ids")
    exp2, _ = orc2.hash_varlen(exp1.reshape(-1)[:T], cu, np.zeros(B2, dtype=np.int64))
    H.assert_bits_equal(h2.cpu().numpy(), exp2, "packed call 2 hash ids (its ids are call 1's output)")
    H.assert_bits_equal(H.bf16_bits(out2[0]), H.oracle_lookup_rows(wl, 0, exp2[:, 0, :]), "packed call 2 rows")
    st1.status()
    st2.status()

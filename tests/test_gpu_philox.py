"""GPU parity of dflash2_philox_uniforms against the oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
from block_draft_proposal_gb300 import dflash2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed,offset,n", [
    (0, 0, 1), (0x5EED, 7, 5), (2**64 - 1, 2**40 + 3, 480), (12345, 99, 7681),
    (42, 2**63 + 11, 1 << 20),
])
def test_uniforms_match_oracle(cuda, seed, offset, n):
    got = dflash2.philox_uniforms(seed, n, offset=offset, device=cuda)
    np.testing.assert_array_equal(got.cpu().numpy(), oracle.philox_uniforms(seed, offset, n))


def test_unaligned_output(cuda):
    buf = torch.zeros(1 + 103, dtype=torch.float32, device=cuda)
    out = buf[1:]  # 4-byte aligned, not 16: the scalar store path
    dflash2.philox_uniforms(9, 103, out=out, offset=5)
    np.testing.assert_array_equal(out.cpu().numpy(), oracle.philox_uniforms(9, 5, 103))
    assert buf[0].item() == 0.0


def test_device_counter_advances(cuda):
    c0 = 2**40 + 3
    counter = torch.tensor([c0], dtype=torch.int64, device=cuda)
    n = 481
    nb = (n + 3) // 4
    a = dflash2.philox_uniforms(77, n, counter=counter, offset=2).cpu().numpy()
    b = dflash2.philox_uniforms(77, n, counter=counter, offset=2).cpu().numpy()
    np.testing.assert_array_equal(a, oracle.philox_uniforms(77, c0 + 2, n))
    np.testing.assert_array_equal(b, oracle.philox_uniforms(77, c0 + nb + 2, n))
    assert counter.item() == c0 + 2 * nb


def test_graph_replay_draws_fresh_sequences(cuda):
    n, seed, c0 = 480, 0xC0FFEE, 1000
    counter = torch.tensor([c0], dtype=torch.int64, device=cuda)
    out = torch.empty(n, dtype=torch.float32, device=cuda)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dflash2.philox_uniforms(seed, n, out=out, counter=counter, stream=s)  # warm-up call
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dflash2.philox_uniforms(seed, n, out=out, counter=counter,
                                stream=torch.cuda.current_stream())
    nb = (n + 3) // 4
    start = counter.item()  # capture does not run the kernel
    assert start == c0 + nb
    for r in range(3):
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(),
                                      oracle.philox_uniforms(seed, start + r * nb, n))
    assert counter.item() == start + 3 * nb


def test_argument_errors(cuda):
    counter = torch.tensor([5], dtype=torch.int64, device=cuda)
    out = torch.empty(8, dtype=torch.float32, device=cuda)
    lib = dflash2.library()
    assert lib.dflash2_philox_uniforms(1, 0, None, -1, out.data_ptr(), None) == 1
    assert lib.dflash2_philox_uniforms(1, 0, None, 4, None, None) == 1
    assert lib.dflash2_philox_uniforms(1, 0, counter.data_ptr(), (1 << 24) + 1, out.data_ptr(),
                                       None) == 1
    assert lib.dflash2_philox_uniforms(1, 0, counter.data_ptr(), 0, out.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert counter.item() == 5


def test_step_with_device_uniforms_in_graph(cuda):
    from block_draft_proposal_gb300 import synth
    w = synth.BY_NAME["qwen3-8b-bf16"].scaled(batch=4, draft_vocab=20000, target_vocab=20000,
                                             sampling="sampled")
    inp = synth.make(w)
    t = {k: dflash2.to_device(v, cuda) for k, v in inp.items() if v is not None}
    bufs = dflash2.ProposalBuffers(w, cuda)
    counter = torch.zeros(1, dtype=torch.int64, device=cuda)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        dflash2.proposal_step(w, t, bufs, stream=s, rng=(w.seed, counter))  # warm-up
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            dflash2.proposal_step(w, t, bufs, stream=s, rng=(w.seed, counter))
    nb = (w.rows + 3) // 4
    base = counter.item()
    for r in range(3):
        g.replay()
        torch.cuda.synchronize()
        want_u = oracle.philox_uniforms(w.seed, base + r * nb, w.rows)
        np.testing.assert_array_equal(bufs.uniforms.cpu().numpy().reshape(-1), want_u)
        # the walk consumed exactly these uniforms: an eager walk on the same
        # candidates and uniforms gives the same tokens and q, bit for bit
        u_dev = torch.from_numpy(want_u.reshape(w.batch, w.slots)).to(cuda)
        tok, q, _, err = dflash2.selector_walk(
            t["h"], t["proj"], t["A"], t["B"], t["anchors"],
            bufs.cand_ids.view(w.batch, w.slots, w.top_k),
            bufs.cand_u.view(w.batch, w.slots, w.top_k), t["temperatures"], t["greedy"], u_dev)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(tok, bufs.tokens) and torch.equal(q, bufs.q)
    assert counter.item() == base + 3 * nb

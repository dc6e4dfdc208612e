"""GPU parity of dflash2_d2t_remap (bit-exact), and of the whole proposal step
end to end (conv, candidates, walk, remap) against the chained oracle,
including replay from a captured CUDA graph."""
import numpy as np
import pytest
import torch

import oracle
from block_draft_proposal_gb300 import dflash2, synth
from parity import check_step_against_oracle

pytestmark = pytest.mark.gpu


def test_d2t_identity_and_padded_ids(cuda):
    ids = torch.tensor([0, 5, 199, 200, 250, -1], dtype=torch.int64, device=cuda)
    out, err = dflash2.d2t_remap(ids, None, draft_vocab=256, target_vocab=200)
    torch.cuda.synchronize()
    ref, nerr = oracle.d2t(ids.cpu().numpy(), None, 256, 200)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)
    assert nerr == 3 and int(err.item()) & dflash2.DEVERR_ID_RANGE


def test_d2t_table_matches_oracle_bit_exact(cuda):
    w = synth.BY_NAME["reduced-vocab-bs12-bf16"]
    table = synth.d2t_table(w)
    rng = np.random.default_rng(110)
    ids = rng.integers(0, w.draft_vocab, size=100_003).astype(np.int64)
    ids[::997] = w.draft_vocab + 3                          # sprinkle invalid ids
    t_ids = torch.from_numpy(ids).to(cuda)
    out, err = dflash2.d2t_remap(t_ids, torch.from_numpy(table).to(cuda), w.draft_vocab,
                                 w.target_vocab)
    torch.cuda.synchronize()
    ref, nerr = oracle.d2t(ids, table, w.draft_vocab, w.target_vocab)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)
    assert nerr > 0 and int(err.item()) & dflash2.DEVERR_ID_RANGE
    # in place
    dflash2.d2t_remap(t_ids, torch.from_numpy(table).to(cuda), w.draft_vocab, w.target_vocab,
                      out=t_ids)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(t_ids.cpu().numpy(), ref)


@pytest.mark.parametrize("name,scale", [("tiny-fp32", {}),
                                        ("reduced-vocab-bs12-bf16", dict(batch=6)),
                                        ("padded-vocab-bf16", dict(batch=2)),
                                        ("stress-bf16", dict(batch=3, draft_vocab=40000,
                                                             target_vocab=40000))])
def test_proposal_step_end_to_end(cuda, name, scale):
    w = synth.BY_NAME[name].scaled(**scale)
    inp = synth.make(w)
    t = {k: dflash2.to_device(v, cuda) for k, v in inp.items() if v is not None}
    out = dflash2.proposal_step(w, t)
    torch.cuda.synchronize()
    assert int(out["err"].item()) & ~dflash2.DEVINFO_TOPK_FALLBACK == 0
    topk_ties, walk_ties = check_step_against_oracle(w, inp, out)
    print(f"{name}: end-to-end near-ties accepted: top-K {topk_ties}, walk {walk_ties}")


def test_captured_graph_replays_the_eager_step(cuda):
    w = synth.BY_NAME["qwen3-8b-bf16"].scaled(batch=4, draft_vocab=20000, target_vocab=20000)
    inp = synth.make(w)
    t = {k: dflash2.to_device(v, cuda) for k, v in inp.items() if v is not None}
    bufs = dflash2.ProposalBuffers(w, cuda)
    eager = {k: v.clone() for k, v in dflash2.proposal_step(w, t, bufs).items()}
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        dflash2.proposal_step(w, t, bufs)        # warm the stream before capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            dflash2.proposal_step(w, t, bufs)
    for v in (bufs.tokens, bufs.q, bufs.cand_ids):
        v.zero_()
    g.replay()
    torch.cuda.synchronize()
    for key in ("cand_ids", "cand_u", "tokens", "q", "target_ids", "conv_out"):
        assert torch.equal(getattr(bufs, key), eager[key]), key


@pytest.mark.parametrize("name,scale", [("qwen3-8b-bf16", dict(batch=6, draft_vocab=30000,
                                                               target_vocab=30000)),
                                        ("tiny-fp32", {})])
def test_overlapped_step_equals_the_one_stream_step(cuda, name, scale):
    """The conv, the uniforms and the selector projection on a second stream
    beside the top-K change no result: every output equals the one-stream
    step's, bit for bit (the same Philox counter draws the same uniforms)."""
    w = synth.BY_NAME[name].scaled(**scale)
    inp = synth.make(w)
    t = {k: dflash2.to_device(v, cuda) for k, v in inp.items() if v is not None}
    outs = []
    for overlap in (False, True):
        bufs = dflash2.ProposalBuffers(w, cuda)
        counter = torch.zeros(1, dtype=torch.int64, device=cuda)
        out = dflash2.proposal_step(w, t, bufs, rng=(w.seed, counter), overlap=overlap)
        torch.cuda.synchronize()
        outs.append({k: v.clone() for k, v in out.items()})
    for key in ("conv_out", "cand_ids", "cand_u", "tokens", "q", "target_ids", "uniforms", "err"):
        assert torch.equal(outs[0][key], outs[1][key]), key

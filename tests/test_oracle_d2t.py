"""Pins for the oracle's draft-to-target id remap.

vLLM Qwen3DSparkForCausalLM.map_draft_to_target: target = draft + d2t[draft]
(d2t holds offsets); no table means the identity, which is the case exactly
when the draft vocab is not smaller than the target vocab.
"""
import numpy as np

from block_draft_proposal_gb300 import synth


def test_identity_without_table(ora):
    ids = np.array([0, 5, 99, 100, 150], np.int64)
    out, errors = ora.d2t(ids, None, draft_vocab=101, target_vocab=100)
    np.testing.assert_array_equal(out, [0, 5, 99, 0, 0])   # 100 is a padded id
    assert errors == 2




def test_offset_table_maps_onto_the_pruned_subset(ora):
    # build the table from a known sorted subset S: draft id i must map to S[i]
    rng = np.random.default_rng(30)
    vt, vd = 1000, 137
    subset = np.sort(rng.choice(vt, size=vd, replace=False))
    table = subset - np.arange(vd)
    ids = rng.integers(0, vd, size=500)
    out, errors = ora.d2t(ids, table, vd, vt)
    assert errors == 0
    np.testing.assert_array_equal(out, subset[ids])
    mapped, _ = ora.d2t(np.arange(vd), table, vd, vt)
    assert np.all(np.diff(mapped) > 0)


def test_generated_reduced_vocab_table_is_strictly_increasing(ora):
    w = synth.BY_NAME["reduced-vocab-bs12-bf16"]
    table = synth.d2t_table(w)
    assert table.shape == (w.draft_vocab,) and np.all(table >= 0)
    mapped, errors = ora.d2t(np.arange(w.draft_vocab), table, w.draft_vocab, w.target_vocab)
    assert errors == 0 and np.all(np.diff(mapped) > 0) and mapped[-1] < w.target_vocab


def test_range_checks(ora):
    table = np.array([0, 1, 5, 200], np.int64)
    out, errors = ora.d2t(np.array([-1, 0, 3, 4, 2], np.int64), table, 4, 100)
    np.testing.assert_array_equal(out, [0, 0, 0, 0, 7])   # 3 + 200 lands past the target vocab
    assert errors == 3

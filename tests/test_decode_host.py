"""Host logic of the closed-loop driver (drift_aware_kv_gb300/decode.py) with a
stand-in for the context: the order of the five calls per step, block entries
only at the first step of each block, n_unmasked fed back from the previous
step's commits (the tau_upd input of §4.1), the blocks advancing in lockstep
once no sequence has a masked token left, and the App. D.1 tokens-per-forward
accounting.  No GPU: the stand-in commits a scripted number of tokens."""
import types

import pytest

torch = pytest.importorskip("torch")


class FakeContext:
    """Records the calls of decode.Generator; commits `script[block][step]`
    tokens per sequence, each step."""

    def __init__(self, batch, n_blocks, block, script):
        self.w = types.SimpleNamespace(batch=batch, n_blocks=n_blocks, block=block, seq_len=8, d_model=4)
        self.script = script
        self.calls = []
        self.left = None
        self.blk = -1
        self.step_in_block = 0

    def embed(self, embed, mask_emb, tokens, masked, x0):
        self.calls.append(("embed",))

    def calibrate_step(self, x0, n_unmasked, block, entry):
        self.calls.append(("calibrate", block, bool(entry), list(n_unmasked)))
        if entry:
            self.blk = block
            self.step_in_block = 0
            self.left = [self.w.block] * self.w.batch

    def decode_logits(self, lm_head, final_norm, logits):
        self.calls.append(("decode_logits",))

    def commit(self, logits, masked, commit, conf):
        self.calls.append(("commit",))

    def decode_tokens(self, logits, commit, tokens, masked):
        self.calls.append(("decode_tokens",))
        counts = []
        for s in range(self.w.batch):
            c = min(self.script[self.blk][self.step_in_block][s], self.left[s])
            self.left[s] -= c
            counts.append(c)
        self.step_in_block += 1
        return counts, list(self.left)


def _weights():
    t = torch.zeros(4, 4)
    return {"embed": t, "mask_emb": t[0], "lm_head": t, "final_norm": t[0]}


def _gen(ctx):
    from drift_aware_kv_gb300.decode import Generator
    return Generator(ctx, _weights())


def test_blocks_advance_in_lockstep_and_counts_feed_back():
    # two sequences, blocks of 4: block 0 finishes in 2 steps (seq 1 slower:
    # 1 + 3), block 1 in 3 steps (seq 0: 2 + 1 + 1)
    script = [
        [[3, 1], [1, 3], [0, 0]],
        [[2, 4], [1, 0], [1, 0]],
    ]
    ctx = FakeContext(batch=2, n_blocks=2, block=4, script=script)
    tokens = torch.zeros(2, 8, dtype=torch.int32)
    masked = torch.ones(2, 8, dtype=torch.uint8)
    st = _gen(ctx).generate(tokens, masked)
    cal = [c for c in ctx.calls if c[0] == "calibrate"]
    # entries exactly at the first step of each block, blocks in order
    assert [(c[1], c[2]) for c in cal] == [(0, True), (0, False), (1, True), (1, False), (1, False)]
    # n_unmasked: zeros at an entry, else the previous step's commits
    assert [c[3] for c in cal] == [[0, 0], [3, 1], [0, 0], [2, 4], [1, 0]]
    # five calls per step, in order
    names = [c[0] for c in ctx.calls]
    assert names == ["embed", "calibrate", "decode_logits", "commit", "decode_tokens"] * 5
    assert st.steps == 5 and st.block_entries == 2
    assert st.per_block_steps == [2, 3]
    assert st.committed == 2 * 4 * 2  # every generated token of both blocks, both sequences
    assert st.tokens_per_forward(2) == pytest.approx(8 / 5)


def test_steps_iterator_reports_what_is_left():
    script = [[[1, 2], [1, 0]]]
    ctx = FakeContext(batch=2, n_blocks=1, block=2, script=script)
    out = list(_gen(ctx).steps(torch.zeros(2, 8, dtype=torch.int32), torch.ones(2, 8, dtype=torch.uint8)))
    assert [(b, e, c, l) for b, e, c, l in out] == [(0, True, [1, 2], [1, 0]), (0, False, [1, 0], [0, 0])]


def test_block_that_never_finishes_is_an_error():
    # the progress rule guarantees a commit per step on the device; a context
    # that commits nothing must not loop forever
    script = [[[0, 0]] * 3]
    ctx = FakeContext(batch=2, n_blocks=1, block=3, script=script)
    with pytest.raises(RuntimeError, match="still has masked tokens"):
        _gen(ctx).generate(torch.zeros(2, 8, dtype=torch.int32), torch.ones(2, 8, dtype=torch.uint8))

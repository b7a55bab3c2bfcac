"""Closed-loop generation on the device with Polestar calibration and commit
("Polestar: Drift-Aware Cache Calibration and Token Commitment for Efficient
Inference of Diffusion LLMs", Algorithm 1 in full; Eq. 1 greedy
reconstruction; App. D.1 tokens-per-forward accounting).

Every step of a block runs five C-ABI calls on the context's main stream:

  polestar_embed          tokens + mask -> layer-0 inputs x0
  polestar_calibrate_step the layer loop (block entry or within-block step)
  polestar_decode_logits  final norm + LM head over the 2B rows the gate scores
  polestar_commit         confidence, drift gate, suffix commit
  polestar_decode_tokens  progress rule, greedy tokens into the committed
                          positions, per-sequence counts back to the host

Blocks advance in lockstep over the batch: the next block's entry comes once no
sequence has a masked token left in the current block.  The counts that
polestar_decode_tokens returns are the next step's n_unmasked (the tau_upd
trigger of §4.1) and the numerator of tokens per forward.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List

import torch


@dataclasses.dataclass
class GenerationStats:
    steps: int = 0  # forward passes (denoising steps) over the batch
    block_entries: int = 0
    committed: int = 0  # generated tokens committed, all sequences
    per_block_steps: List[int] = dataclasses.field(default_factory=list)

    def tokens_per_forward(self, batch: int) -> float:
        """App. D.1: generated tokens per sequence / forward passes."""
        return self.committed / batch / max(self.steps, 1)


class Generator:
    """Device buffers of one closed loop over a Polestar context.

    decode_weights: "embed" [V, d], "mask_emb" [d], "lm_head" [V, d],
    "final_norm" [d], CUDA tensors in the context's storage dtype."""

    def __init__(self, ps, decode_weights: Dict[str, torch.Tensor]):
        self.ps = ps
        w = ps.w
        self.dw = decode_weights
        V = int(decode_weights["lm_head"].shape[0])
        dev = decode_weights["lm_head"].device
        dt = decode_weights["lm_head"].dtype
        self.V = V
        self.x0 = torch.empty(w.batch, w.seq_len, w.d_model, dtype=dt, device=dev)
        self.logits = torch.empty(w.batch, 2 * w.block, V, dtype=torch.float32, device=dev)
        self.commit = torch.zeros(w.batch, 2 * w.block, dtype=torch.uint8, device=dev)
        self.conf = torch.empty(w.batch, 2 * w.block, dtype=torch.float32, device=dev)

    def step(self, tokens, masked_u8, block: int, entry: bool, n_unmasked):
        """One denoising step; updates tokens [batch, N] int32 and masked_u8
        [batch, N] uint8 in place.  Returns (committed, still masked in the
        block), per sequence."""
        ps, d = self.ps, self.dw
        ps.embed(d["embed"], d["mask_emb"], tokens, masked_u8, self.x0)
        ps.calibrate_step(self.x0, n_unmasked, block, entry)
        ps.decode_logits(d["lm_head"], d["final_norm"], self.logits)
        ps.commit(self.logits, masked_u8, self.commit, self.conf)
        return ps.decode_tokens(self.logits, self.commit, tokens, masked_u8)

    def steps(self, tokens, masked_u8):
        """Iterate the generation step by step (Algorithm 1): yields after every
        step (block index, whether it was the block's entry, per-sequence
        committed counts, per-sequence tokens still masked in the block)."""
        w = self.ps.w
        for blk in range(w.n_blocks):
            entry = True
            n_unmasked = [0] * w.batch
            # the progress rule commits at least one token of the block per step
            for _ in range(w.block):
                counts, left = self.step(tokens, masked_u8, blk, entry, n_unmasked)
                yield blk, entry, counts, left
                n_unmasked = counts
                entry = False
                if max(left) == 0:
                    break
            else:
                raise RuntimeError(f"block {blk} still has masked tokens after {w.block} steps")

    def generate(self, tokens, masked_u8) -> GenerationStats:
        """Decode every block of the generated region (Algorithm 1)."""
        st = GenerationStats()
        steps = 0
        for blk, entry, counts, left in self.steps(tokens, masked_u8):
            if entry and steps:
                st.per_block_steps.append(steps)
                steps = 0
            st.steps += 1
            st.block_entries += int(entry)
            st.committed += sum(counts)
            steps += 1
        if steps:
            st.per_block_steps.append(steps)
        return st

"""Sharded receiver of LoCo's data-parallel step.

"LoCo: Low-Bit Communication Adaptor for Large-scale Model Training", §3.3
(the all-to-all alternative to a reduce-scatter, around Eqn 8) and the
16-bit parameter all-gather of the Table I discussion: each of W ranks
compresses its whole bucket (loco_compress), one all-to-all sends shard j of
every rank's packed codes and steps to rank j, rank j decodes and averages the
W slices it received in fp32 and updates its shard of the parameters
(loco_decode_reduce, loco_adam_step[_bf16] or loco_sgd_step on the shard), and
the updated 16-bit parameter shards are all-gathered.  A partial sum is never
re-compressed, which is why the pages prefer the all-to-all: a reduce-scatter
would decompress, add and compress again at every hop.

The shard map is ``loco_shard_range`` of the C ABI: units of 4*block elements,
so every shard starts on a quant-block boundary and its codes and steps start
16-byte aligned.  The exchanges are ``torch.distributed.all_to_all_single``
calls (NCCL on GPUs, gloo on CPU), one for the codes and one for the steps,
taken straight out of the rank's own buffers (shard j's codes and steps are
contiguous, in shard order), so nothing is packed or copied on the sending
side.  A rank's scales buffer must hold ``scales_capacity(n, block)`` floats
(nb rounded up to a multiple of 4): the last shard's steps travel as whole
16-byte pieces, so every received slice starts 16-byte aligned in the receive
buffer, as the receiver kernels require; the padding steps are never read.

All arithmetic runs in libloco's kernels; this module only sizes buffers,
issues the collectives and passes pointers.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from bit_gradient_compression_gb300 import loco as L


def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def scales_capacity(n: int, block: int) -> int:
    """Floats a rank's scales buffer must hold for the exchange: nb rounded up to 4."""
    return _round_up(L.loco_num_blocks(n, block), 4)


def shard_ranges(n: int, block: int, W: int) -> list[tuple[int, int]]:
    """Element ranges [lo, hi) of the W shards, in rank order."""
    return [L.loco_shard_range(n, block, W, j) for j in range(W)]


class ShardedReceiver:
    """Receive side of one rank of a W-rank group for buckets of n elements.

    After ``exchange(codes, scales)`` the receive buffers hold, for every
    source rank r, the codes and steps of this rank's shard [lo, hi) of rank
    r's bucket; ``slices()`` returns them as W (codes, steps) views, which is
    exactly what loco_decode_reduce / loco_adam_step take for the shard."""

    def __init__(self, n: int, bits: int, block: int, group=None, device=None):
        self.group = group
        self.W = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.n, self.bits, self.block = n, bits, block
        self.ranges = shard_ranges(n, block, self.W)
        self.lo, self.hi = self.ranges[self.rank]
        self.n_shard = self.hi - self.lo
        self.code_splits = [L.loco_code_bytes(h - l, bits, block) for l, h in self.ranges]
        self.scale_splits = [_round_up(L.loco_num_blocks(h - l, block), 4) for l, h in self.ranges]
        self.code_bytes = L.loco_code_bytes(n, bits, block)
        self.scale_floats = scales_capacity(n, block)
        assert sum(self.code_splits) == self.code_bytes and sum(self.scale_splits) == self.scale_floats
        dev = torch.device(device) if device is not None else torch.device("cpu")
        cb, sb = self.code_splits[self.rank], self.scale_splits[self.rank]
        self.recv_codes = torch.empty(self.W * cb, dtype=torch.uint8, device=dev)
        self.recv_scales = torch.empty(self.W * sb, dtype=torch.float32, device=dev)
        # 16-bit parameter all-gather: every rank contributes a slot of the longest shard's length
        self.shard_max = max(h - l for l, h in self.ranges)
        self.bf16_send = torch.empty(self.shard_max, dtype=torch.int16, device=dev)

    # ------------------------------------------------------------------ exchange

    def exchange(self, codes: torch.Tensor, scales: torch.Tensor, async_op: bool = False):
        """All-to-all of the shards of this rank's packed bucket (codes: uint8
        [loco_code_bytes(n)], scales: float32 [>= scales_capacity(n, block)])."""
        if codes.numel() < self.code_bytes or scales.numel() < self.scale_floats:
            raise ValueError(f"codes need {self.code_bytes} bytes and scales {self.scale_floats} floats "
                             f"(got {codes.numel()} and {scales.numel()})")
        cb, sb = self.code_splits[self.rank], self.scale_splits[self.rank]
        w1 = dist.all_to_all_single(self.recv_codes, codes[:self.code_bytes], [cb] * self.W, self.code_splits,
                                    group=self.group, async_op=async_op)
        w2 = dist.all_to_all_single(self.recv_scales, scales[:self.scale_floats], [sb] * self.W, self.scale_splits,
                                    group=self.group, async_op=async_op)
        return (w1, w2) if async_op else None

    def slices(self):
        """W views (source rank order) of the received codes and steps of this shard."""
        cb, sb = self.code_splits[self.rank], self.scale_splits[self.rank]
        codes = [self.recv_codes[r * cb:(r + 1) * cb] for r in range(self.W)]
        scales = [self.recv_scales[r * sb:(r + 1) * sb] for r in range(self.W)]
        return codes, scales

    # ------------------------------------------------------------------ shard-local receiver steps

    def shard(self, t: torch.Tensor) -> torch.Tensor:
        """This rank's shard [lo, hi) of a full-length tensor (a view)."""
        return t[self.lo:self.hi]

    def decode_reduce(self, cfg, mean_shard, stream=None):
        codes, scales = self.slices()
        L.loco_decode_reduce(cfg, codes, scales, self.n_shard, mean_shard, stream=stream)

    def adam_step(self, cfg, param_shard, m_shard, v_shard, hp, t: int, bf16: bool = False, stream=None):
        """Fused average + Adam(W) on this shard; with bf16, the rounded copy of the
        updated shard goes to the all-gather slot (see gather_params_bf16)."""
        codes, scales = self.slices()
        if bf16:
            L.loco_adam_step_bf16(cfg, codes, scales, self.n_shard, param_shard, m_shard, v_shard,
                                  self.bf16_send[:self.n_shard], hp, t, stream=stream)
        else:
            L.loco_adam_step(cfg, codes, scales, self.n_shard, param_shard, m_shard, v_shard, hp, t, stream=stream)

    def sgd_step(self, cfg, param_shard, lr: float, bf16: bool = False, stream=None):
        codes, scales = self.slices()
        L.loco_sgd_step(cfg, codes, scales, self.n_shard, param_shard, lr,
                        param_bf16=self.bf16_send[:self.n_shard] if bf16 else None, stream=stream)

    # ------------------------------------------------------------------ 16-bit parameter all-gather

    def gather_params_bf16(self, out: torch.Tensor | None = None) -> torch.Tensor:
        """All-gather of every rank's bf16 parameter shard (the slot filled by a
        bf16 optimizer step) into ``out`` [W * shard_max] (int16 bit patterns):
        rank j's shard is out[j*shard_max : j*shard_max + (hi_j - lo_j)]."""
        if out is None:
            out = torch.empty(self.W * self.shard_max, dtype=torch.int16, device=self.bf16_send.device)
        # moved as bytes: every backend carries uint8
        raw, slot = out.view(torch.uint8), 2 * self.shard_max
        slots = [raw[j * slot:(j + 1) * slot] for j in range(self.W)]
        dist.all_gather(slots, self.bf16_send.view(torch.uint8), group=self.group)
        return out

    def unpad(self, gathered: torch.Tensor) -> torch.Tensor:
        """The full bucket's bf16 parameters [n] from a gather_params_bf16 result
        (a view when every shard has the same length)."""
        if all(h - l == self.shard_max for l, h in self.ranges):
            return gathered[:self.n]
        return torch.cat([gathered[j * self.shard_max:j * self.shard_max + (h - l)]
                          for j, (l, h) in enumerate(self.ranges)])

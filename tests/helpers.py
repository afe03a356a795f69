"""Shared test utilities: host copies of device buffers and sampled comparisons."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def grad_to_np(t: torch.Tensor) -> np.ndarray:
    """Host copy of a gradient: float32 array, or uint16 bf16 bit patterns."""
    c = t.detach().cpu()
    if c.dtype == torch.bfloat16:
        return c.view(torch.int16).numpy().view(np.uint16).copy()
    return c.numpy().copy()


def np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().copy()


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str):
    if got.dtype == np.float32:
        g, w = got.view(np.uint32), want.view(np.uint32)
    else:
        g, w = got, want
    bad = np.nonzero(g != w)[0]
    assert bad.size == 0, f"{what}: {bad.size} mismatches, first at {bad[:5]}: got {got[bad[:5]]} want {want[bad[:5]]}"


def sample_block_ids(nb: int, count: int, seed: int) -> np.ndarray:
    """First, last and `count` random quant blocks (sorted, unique)."""
    rng = np.random.default_rng(seed)
    ids = set([0, nb - 1])
    ids.update(int(x) for x in rng.integers(0, nb, size=count))
    return np.array(sorted(ids), dtype=np.int64)


def gather_blocks(t: torch.Tensor, block_ids: np.ndarray, block: int, n: int) -> list:
    """Host copies of the elements of each listed quant block of a flat tensor."""
    out = []
    for b in block_ids:
        lo = int(b) * block
        hi = min(lo + block, n)
        out.append(t[lo:hi])
    cat = torch.cat(out).cpu()
    res, off = [], 0
    for b in block_ids:
        cnt = min(int(b) * block + block, n) - int(b) * block
        res.append(cat[off:off + cnt])
        off += cnt
    return res


def gather_code_blocks(codes: torch.Tensor, block_ids, block: int, bits: int) -> list:
    bpb = block * bits // 8
    idx = torch.as_tensor(block_ids, device=codes.device)
    rows = codes.view(-1, bpb).index_select(0, idx).cpu().numpy()
    return [rows[i].copy() for i in range(rows.shape[0])]


def oracle_compress_blocks(g_blocks, e_blocks, step, *, bits, block, **kw):
    """Run the oracle on each sampled block as its own bucket; returns codes, scales, new e per block."""
    out = []
    for gb, eb in zip(g_blocks, e_blocks):
        g = grad_to_np(gb) if isinstance(gb, torch.Tensor) else gb
        e = eb.numpy().copy() if isinstance(eb, torch.Tensor) else eb.copy()
        c, s = oracle.compress(g, e, step, bits=bits, block=block, **kw)
        out.append((c, s, e))
    return out


def block_index(ids: np.ndarray, block: int, n: int, device) -> torch.Tensor:
    """Element indices of the listed quant blocks, concatenated (ragged last block clipped)."""
    idx = (torch.as_tensor(ids, device=device)[:, None] * block + torch.arange(block, device=device)[None, :]).reshape(-1)
    return idx[idx < n]


def take(t: torch.Tensor, idx: torch.Tensor) -> torch.Tensor:
    """Host copy of t[idx]."""
    return t.index_select(0, idx).cpu()


def code_rows(codes: torch.Tensor, ids: np.ndarray, block: int, bits: int) -> np.ndarray:
    bpb = block * bits // 8
    return codes.view(-1, bpb).index_select(0, torch.as_tensor(ids, device=codes.device)).cpu().numpy().reshape(-1)


def scale_rows(scales: torch.Tensor, ids: np.ndarray) -> np.ndarray:
    return scales.index_select(0, torch.as_tensor(ids, device=scales.device)).cpu().numpy()


class Stage:
    """Page-locked host buffers, reused by name, for chunked whole-bucket
    comparisons: fetch() copies a device slice into one and returns it as a
    numpy array (valid until the next fetch under the same name); put() copies
    a numpy view of a stage buffer back into device storage."""

    def __init__(self):
        self.bufs = {}

    def _buf(self, name: str, nbytes: int) -> torch.Tensor:
        b = self.bufs.get(name)
        if b is None or b.numel() < nbytes:
            b = torch.empty(max(nbytes, 16), dtype=torch.uint8, pin_memory=True)
            self.bufs[name] = b
        return b[:nbytes]

    def fetch(self, name: str, t: torch.Tensor, np_dtype) -> np.ndarray:
        nbytes = t.numel() * t.element_size()
        b = self._buf(name, nbytes)
        b.copy_(t.reshape(-1).view(torch.uint8), non_blocking=True)
        torch.cuda.current_stream().synchronize()
        return b.numpy().view(np_dtype)

    def zeros(self, name: str, count: int, np_dtype) -> np.ndarray:
        a = self._buf(name, count * np.dtype(np_dtype).itemsize).numpy().view(np_dtype)
        a[:] = 0
        return a

    def array(self, name: str, count: int, np_dtype) -> np.ndarray:
        return self._buf(name, count * np.dtype(np_dtype).itemsize).numpy().view(np_dtype)

    def put(self, dst: torch.Tensor, arr: np.ndarray):
        src = torch.from_numpy(arr.view(np.uint8))
        dst.reshape(-1).view(torch.uint8).copy_(src, non_blocking=True)
        torch.cuda.current_stream().synchronize()

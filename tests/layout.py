"""Read a cache buffer back into the oracle's per-position arrays (test helper, layout only).

Follows the buffer layout documented in include/kvq.h: 256-byte aligned regions, the header first,
then ring_k, ring_v and the pages; the offsets below are derived from the end of the buffer, which
is exactly the pages region.  No arithmetic of the method happens here -- only bit unpacking.
"""

from __future__ import annotations

import numpy as np
import torch

P = 64      # tokens per page (block-table granularity)
H = 32      # tokens per half-page (one contiguous set of regions)


def _a256(x: int) -> int:
    return (x + 255) & ~255


def regions(cfg, total: int) -> dict:
    kmain = {1: 64, 3: 64, 4: 128}[cfg.k_format]        # K main bytes per token: Q4G32, TQ3_QJL, Q8G32
    kmeta = {1: 16, 3: 4, 4: 8}[cfg.k_format]
    half_bytes = (kmain + 64) * H + kmeta * H + 16 * H  # K main | V main | K meta | V meta (32 tokens)
    page_bytes = 2 * half_bytes
    maxpps = -(-cfg.max_seq_len // P)
    n_pages = cfg.n_pages or cfg.max_batch * maxpps
    pages = cfg.n_layers * n_pages * cfg.n_kv_heads * page_bytes
    assert pages % 256 == 0
    off_pages = total - pages
    ring = _a256(cfg.n_layers * cfg.max_batch * cfg.n_kv_heads * cfg.window * 128 * 4)
    off_ringv = off_pages - ring
    off_ringk = off_ringv - ring
    off_bt = off_ringk - _a256(cfg.max_batch * maxpps * 4)
    sig = _a256(cfg.n_layers * cfg.n_kv_heads * 128 * 2)
    off_sigv = off_bt - sig
    off_sigk = off_sigv - sig
    return dict(page_bytes=page_bytes, half_bytes=half_bytes, n_pages=n_pages, maxpps=maxpps,
                off_pages=off_pages, off_ringk=off_ringk, off_ringv=off_ringv, off_sigk=off_sigk,
                off_sigv=off_sigv, kmain=kmain, kmeta=kmeta, off_bt=off_bt)


def _gather(buf: torch.Tensor, starts: np.ndarray, n: int) -> np.ndarray:
    idx = torch.as_tensor(starts, dtype=torch.int64, device=buf.device)[:, None] + \
        torch.arange(n, dtype=torch.int64, device=buf.device)[None, :]
    return buf[idx.reshape(-1)].reshape(len(starts), n).cpu().numpy()


def _q4k_codes(rec: np.ndarray) -> np.ndarray:
    """K record [T][64]: word (i, G) at byte 16i + 4G holds channels 32G + 8i .. +7, byte k = channels
    32G + 8i + 2k (low nibble) and + 1 (high nibble)."""
    b = rec.reshape(-1, 4, 4, 4)                                # [T][i][G][k]
    nib = np.stack([b & 15, b >> 4], axis=-1)                   # [T][i][G][k][lo/hi]
    return nib.transpose(0, 2, 1, 3, 4).reshape(-1, 128).astype(np.uint8)   # channel 32G + 8i + 2k + e


def _q4v_codes(half_v: np.ndarray, t: np.ndarray) -> np.ndarray:
    """V codes of tokens t from the V region of their half-pages (half_v [T][2048] bytes): tokens 2p and
    2p+1 share 128 bytes; row r of group G is at 16*((r + 2*(p & 3)) & 7) + 4G with bytes
    [t0 byte0, t1 byte0, t0 byte1, t1 byte1]; byte0 = channels 32G+4r (low), +1; byte1 = +2, +3."""
    p = t // 2
    slot = t % 2
    out = np.zeros((len(t), 128), np.uint8)
    for r in range(8):
        blk = 16 * ((r + 2 * (p & 3)) & 7)
        for G in range(4):
            base = p * 128 + blk + 4 * G + slot
            b0 = half_v[np.arange(len(t)), base]
            b1 = half_v[np.arange(len(t)), base + 2]
            c = 32 * G + 4 * r
            out[:, c], out[:, c + 1] = b0 & 15, b0 >> 4
            out[:, c + 2], out[:, c + 3] = b1 & 15, b1 >> 4
    return out


def _q8k_codes(rec: np.ndarray, t: np.ndarray) -> np.ndarray:
    """Q8G32 K record [T][128] of tokens with index t in their half-page: 16-byte chunk m = 2i + h at
    16 (m ^ (t & 1)); byte b of its word w = channel 16 (4h + w) + 2i + (b & 1) + 8 (b >> 1); stored
    bytes u = c + 128."""
    out = np.zeros((len(t), 128), np.int8)
    for m in range(8):
        i, h = m >> 1, m & 1
        pos = 16 * (m ^ (t & 1))
        for w in range(4):
            for b in range(4):
                ch = 16 * (4 * h + w) + 2 * i + (b & 1) + 8 * (b >> 1)
                out[:, ch] = (rec[np.arange(len(t)), pos + 4 * w + b].astype(np.int16) - 128).astype(np.int8)
    return out


def _tq3_fields(rec: np.ndarray):
    """TQ3 key record [T][64]: byte j holds the 3-bit codes of channels 2j (bits 0-2) and 2j + 1
    (bits 3-5) and the QJL sign bits of projections 2j (bit 6) and 2j + 1 (bit 7)."""
    codes = np.stack([rec & 7, (rec >> 3) & 7], axis=-1).reshape(-1, 128).astype(np.uint8)
    bits = np.stack([(rec >> 6) & 1, rec >> 7], axis=-1).reshape(-1, 128).astype(bool)
    return codes, bits


def read_unit(buf: torch.Tensor, cfg, layer: int, b: int, h: int, n_tokens: int,
              block_table: np.ndarray | None = None) -> dict:
    """Quantised records of positions [0, n_tokens) of one (layer, sequence, kv-head)."""
    R = regions(cfg, buf.numel())
    if block_table is None:
        block_table = np.arange(cfg.max_batch * R["maxpps"]).reshape(cfg.max_batch, R["maxpps"])
    pos = np.arange(n_tokens)
    phys = block_table[b, pos // P].astype(np.int64)
    base = (R["off_pages"] + ((layer * R["n_pages"] + phys) * cfg.n_kv_heads + h) * R["page_bytes"] +
            ((pos % P) // H) * R["half_bytes"])           # the half-page holding each position
    t = pos % H
    out = {}
    vmain0 = base + R["kmain"] * H
    kmeta0 = vmain0 + 64 * H
    vmeta0 = kmeta0 + R["kmeta"] * H
    if cfg.k_format == 3:
        out["k_code"], out["k_bits"] = _tq3_fields(_gather(buf, base + t * 64, 64))
        out["k_norm"] = _gather(buf, kmeta0 + t * 2, 2).view(np.float16)[:, 0]
        out["k_gamma"] = _gather(buf, kmeta0 + 2 * H + t * 2, 2).view(np.float16)[:, 0]
    elif cfg.k_format == 4:
        out["k_code"] = _q8k_codes(_gather(buf, base + t * 128, 128), t)
        out["k_scale"] = _gather(buf, kmeta0 + t * 8, 8).view(np.float16)
    else:
        out["k_code"] = _q4k_codes(_gather(buf, base + t * 64, 64))
        m = _gather(buf, kmeta0 + t * 16, 16).view(np.float16)
        out["k_scale"], out["k_zero"] = m[:, :4], m[:, 4:]
    out["v_code"] = _q4v_codes(_gather(buf, vmain0, 64 * H), t)
    sc = np.stack([_gather(buf, vmeta0 + (G * H + t) * 2, 2).view(np.float16)[:, 0] for G in range(4)], 1)
    zr = np.stack([_gather(buf, vmeta0 + 8 * H + (G * H + t) * 2, 2).view(np.float16)[:, 0] for G in range(4)], 1)
    out["v_scale"], out["v_zero"] = sc, zr
    return out


def read_ring(buf: torch.Tensor, cfg, layer: int, b: int, h: int):
    R = regions(cfg, buf.numel())
    n = cfg.window * 128 * 4
    o = (((layer * cfg.max_batch + b) * cfg.n_kv_heads + h) * cfg.window) * 128 * 4
    k = buf[R["off_ringk"] + o: R["off_ringk"] + o + n].cpu().numpy().view(np.float32).reshape(cfg.window, 128)
    v = buf[R["off_ringv"] + o: R["off_ringv"] + o + n].cpu().numpy().view(np.float32).reshape(cfg.window, 128)
    return k, v


def read_sigma(buf: torch.Tensor, cfg):
    R = regions(cfg, buf.numel())
    n = cfg.n_layers * cfg.n_kv_heads * 128 * 2
    sk = buf[R["off_sigk"]: R["off_sigk"] + n].cpu().numpy().view(np.float16).reshape(cfg.n_layers, cfg.n_kv_heads, 128)
    sv = buf[R["off_sigv"]: R["off_sigv"] + n].cpu().numpy().view(np.float16).reshape(cfg.n_layers, cfg.n_kv_heads, 128)
    return sk, sv

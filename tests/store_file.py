"""The store file format, written out from its description in kvi.h (file
format, version 1) without any of the library's code: a writer, a reader and
the two hashes.  The tests use it to read files the library wrote and to
build valid and damaged files for the library to read."""
from __future__ import annotations

import struct

import numpy as np

MAGIC = b"KVISTORE"
VERSION = 1
HEADER_BYTES = 128
ALIGN = 4096
FNV_BASIS = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK = (1 << 64) - 1


def fnv1a(data: bytes, h: int = FNV_BASIS) -> int:
    for b in data:
        h = ((h ^ b) * FNV_PRIME) & MASK
    return h


def payload_hash(data: bytes) -> int:
    """Four lanes over little-endian 64-bit words (word i -> lane i mod 4)."""
    words = np.frombuffer(data, dtype="<u8").tolist()
    h = [(FNV_BASIS + j) & MASK for j in range(4)]
    for i, w in enumerate(words):
        j = i & 3
        h[j] = ((h[j] ^ w) * FNV_PRIME) & MASK

    def rotl(x, r):
        return ((x << r) | (x >> (64 - r))) & MASK

    return h[0] ^ rotl(h[1], 16) ^ rotl(h[2], 32) ^ rotl(h[3], 48)


def _up(x: int) -> int:
    return (x + ALIGN - 1) // ALIGN * ALIGN


def layout(g, n: int, t: int) -> dict:
    L, H, D, E = g
    emb = n * E * 4
    kv = L * 2 * t * H * D * 2
    start = _up(HEADER_BYTES)
    ln = _up(start + 8 * n)
    e = _up(ln + 4 * n)
    k = _up(e + emb)
    return {"start": start, "len": ln, "emb": e, "kv": k, "file": k + kv, "emb_bytes": emb, "kv_bytes": kv}


def build(g, fact_start, fact_len, emb: bytes, kv: bytes, n_tokens: int, *, version=VERSION,
          magic=MAGIC, extents_hash=None, payload=None, header_hash=None, offsets=None,
          reserved=b"\0" * 16) -> bytes:
    """Bytes of a store file; the keyword arguments override a field to make
    a damaged file."""
    fs = np.asarray(fact_start, dtype="<i8").tobytes()
    fl = np.asarray(fact_len, dtype="<i4").tobytes()
    n = len(fact_len)
    lay = layout(g, n, n_tokens)
    assert len(emb) == lay["emb_bytes"] and len(kv) == lay["kv_bytes"]
    offs = offsets or [lay["start"], lay["len"], lay["emb"], lay["kv"], lay["file"]]
    eh = fnv1a(fl, fnv1a(fs)) if extents_hash is None else extents_hash
    ph = payload_hash(emb + kv) if payload is None else payload
    head = magic + struct.pack("<II", version, HEADER_BYTES) + struct.pack("<4i", *g)
    head += struct.pack("<qq", n, n_tokens) + struct.pack("<5Q", *offs) + struct.pack("<QQ", eh, ph)
    assert len(head) == 104
    hh = fnv1a(head) if header_hash is None else header_hash
    head += struct.pack("<Q", hh) + reserved
    out = bytearray(lay["file"])
    out[:HEADER_BYTES] = head
    out[lay["start"]:lay["start"] + len(fs)] = fs
    out[lay["len"]:lay["len"] + len(fl)] = fl
    out[lay["emb"]:lay["emb"] + len(emb)] = emb
    out[lay["kv"]:lay["kv"] + len(kv)] = kv
    return bytes(out)


def read(path: str) -> dict:
    """Parse a store file (no checks beyond the layout): header fields and
    the four sections as bytes."""
    data = open(path, "rb").read()
    h = data[:HEADER_BYTES]
    g = struct.unpack_from("<4i", h, 16)
    n, t = struct.unpack_from("<qq", h, 32)
    offs = struct.unpack_from("<5Q", h, 48)
    eh, ph, hh = struct.unpack_from("<QQQ", h, 88)
    lay = layout(g, n, t)
    return {
        "magic": h[:8], "version": struct.unpack_from("<I", h, 8)[0],
        "header_bytes": struct.unpack_from("<I", h, 12)[0], "g": g, "n": n, "t": t,
        "offsets": offs, "extents_hash": eh, "payload_hash": ph, "header_hash": hh,
        "header_hash_ok": fnv1a(h[:104]) == hh, "reserved": h[112:128], "size": len(data),
        "layout": lay,
        "fact_start": data[lay["start"]:lay["start"] + 8 * n],
        "fact_len": data[lay["len"]:lay["len"] + 4 * n],
        "emb": data[lay["emb"]:lay["emb"] + lay["emb_bytes"]],
        "kv": data[lay["kv"]:lay["kv"] + lay["kv_bytes"]],
        "gaps_zero": all(not any(data[a:b]) for a, b in [
            (HEADER_BYTES, lay["start"]), (lay["start"] + 8 * n, lay["len"]),
            (lay["len"] + 4 * n, lay["emb"]), (lay["emb"] + lay["emb_bytes"], lay["kv"])]),
    }

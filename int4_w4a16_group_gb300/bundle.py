"""Writer of the library's multi-tensor weight bundle (the format is stated in w4a16.h, above
w4a16_bundle_info): named (qw [K/8, N] int32, sc [K/32, N] float32) pairs in one file that
w4a16_bundle_load brings onto the device and registers by name. Host-only (numpy)."""
import struct

import numpy as np

MAGIC = b"W4A16BDL"
VERSION = 1
GROUP = 32


def write_bundle(path, tensors) -> None:
    """tensors: mapping (or sequence of pairs) name -> (qw, sc). Blobs start at 16-byte
    aligned file offsets, in the given order."""
    items = list(tensors.items()) if hasattr(tensors, "items") else list(tensors)
    index, blobs = [], []
    for name, (qw, sc) in items:
        qw = np.ascontiguousarray(qw, dtype=np.int32)
        sc = np.ascontiguousarray(sc, dtype=np.float32)
        K8, N = qw.shape
        K = 8 * K8
        if K % GROUP or N % 4 or sc.shape != (K // GROUP, N):
            raise ValueError(f"{name}: qw {qw.shape} / sc {sc.shape} are not a K%32, N%4 pair")
        index.append((name.encode(), K, N))
        blobs.append((qw.tobytes(), sc.tobytes()))
    head = len(MAGIC) + 8 + sum(4 + len(n) + 4 + 4 + 8 + 8 for n, _, _ in index)
    off = (head + 15) & ~15
    offsets = []
    for q, s in blobs:
        qo = off
        off = (off + len(q) + 15) & ~15
        so = off
        off = (off + len(s) + 15) & ~15
        offsets.append((qo, so))
    with open(path, "wb") as f:
        f.write(MAGIC + struct.pack("<II", VERSION, len(index)))
        for (name, K, N), (qo, so) in zip(index, offsets):
            f.write(struct.pack("<I", len(name)) + name + struct.pack("<iiQQ", K, N, qo, so))
        for (q, s), (qo, so) in zip(blobs, offsets):
            f.seek(qo)
            f.write(q)
            f.seek(so)
            f.write(s)
        f.truncate(off)

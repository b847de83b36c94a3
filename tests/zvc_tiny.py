"""An independent pure-Python ZVC codec for tiny inputs (brute force, lists and struct).

Written separately from the C oracle and sharing nothing with it, so that the two can
check each other. Rule: Rhu et al., "Compressing DMA Engine", section V.A (32-word
window, 32-bit zero/non-zero mask, then the non-zero words). The framing follows the
stream layout documented in oracle/zvc_oracle.c.
"""
import itertools
import struct


def tiny_encode(words, chunk_elems):
    words = [int(v) & 0xFFFFFFFF for v in words]
    n = len(words)
    chunks = []
    for c0 in range(0, n, chunk_elems):
        seg = words[c0:c0 + chunk_elems]
        body = []
        for k in range(0, len(seg), 32):
            win = seg[k:k + 32]
            present = [i for i, v in enumerate(win) if v != 0]
            body.append(struct.pack("<I", sum(1 << i for i in present)))
            body.extend(struct.pack("<I", win[i]) for i in present)
        chunks.append(b"".join(body))
    offsets = list(itertools.accumulate([len(b) for b in chunks], initial=0))[:-1]
    payload = b"".join(chunks)
    header = struct.pack("<IHHIIQQ", 0x3143565A, 1, 4, 32, chunk_elems, n, len(payload))
    return header + b"".join(struct.pack("<Q", o) for o in offsets) + payload


def tiny_decode(stream, n, chunk_elems):
    """Returns the words, or None if the stream is not a valid encoding of n words."""
    stream = bytes(stream)
    if len(stream) < 32:
        return None
    magic, ver, wb, win, c, nn, pay = struct.unpack_from("<IHHIIQQ", stream, 0)
    if (magic, ver, wb, win, c, nn) != (0x3143565A, 1, 4, 32, chunk_elems, n):
        return None
    nc = -(-n // chunk_elems)
    base = 32 + 8 * nc
    if len(stream) != base + pay:
        return None
    offs = [struct.unpack_from("<Q", stream, 32 + 8 * i)[0] for i in range(nc)] + [pay]
    out = []
    for ci in range(nc):
        pos, end = offs[ci], offs[ci + 1]
        if (ci == 0 and pos != 0) or not (pos <= end <= pay):
            return None
        count = min(chunk_elems, n - ci * chunk_elems)
        for k in range(0, count, 32):
            if pos + 4 > end:
                return None
            (mask,) = struct.unpack_from("<I", stream, base + pos)
            pos += 4
            valid = min(32, count - k)
            if mask >> valid:
                return None
            for i in range(valid):
                if (mask >> i) & 1:
                    if pos + 4 > end:
                        return None
                    out.append(struct.unpack_from("<I", stream, base + pos)[0])
                    pos += 4
                else:
                    out.append(0)
        if pos != end:
            return None
    return out


def tiny_encode_batch(list_of_words, chunk_elems):
    streams = [tiny_encode(w, chunk_elems) for w in list_of_words]
    head = 16 + 8 * (len(streams) + 1)
    offs = list(itertools.accumulate([len(s) for s in streams], initial=head))
    return (struct.pack("<IIQ", 0x4243565A, len(streams), offs[-1])
            + b"".join(struct.pack("<Q", o) for o in offs) + b"".join(streams))


# ---- ZVC on 16-bit words: the same rule with 2-byte values (word_bytes 2 in the header)
def tiny_encode16(words, chunk_elems):
    words = [int(v) & 0xFFFF for v in words]
    n = len(words)
    bodies = []
    for c0 in range(0, n, chunk_elems):
        seg = words[c0:c0 + chunk_elems]
        parts = []
        for k in range(0, len(seg), 32):
            win = seg[k:k + 32]
            mask = 0
            vals = b""
            for i, v in enumerate(win):
                if v:
                    mask |= 1 << i
                    vals += struct.pack("<H", v)
            parts.append(struct.pack("<I", mask) + vals)
        bodies.append(b"".join(parts))
    offs = list(itertools.accumulate([len(b) for b in bodies], initial=0))[:-1]
    payload = b"".join(bodies)
    head = struct.pack("<IHHIIQQ", 0x3143565A, 1, 2, 32, chunk_elems, n, len(payload))
    return head + b"".join(struct.pack("<Q", o) for o in offs) + payload


def tiny_decode16(stream, n, chunk_elems):
    """Returns the 16-bit words, or None if the stream is not a valid encoding of n."""
    stream = bytes(stream)
    if len(stream) < 32:
        return None
    if struct.unpack_from("<IHHIIQ", stream, 0) != (0x3143565A, 1, 2, 32, chunk_elems, n):
        return None
    (pay,) = struct.unpack_from("<Q", stream, 24)
    nc = -(-n // chunk_elems)
    base = 32 + 8 * nc
    if len(stream) != base + pay:
        return None
    offs = [struct.unpack_from("<Q", stream, 32 + 8 * i)[0] for i in range(nc)] + [pay]
    out = []
    for ci in range(nc):
        pos, end = offs[ci], offs[ci + 1]
        if (ci == 0 and pos != 0) or not (pos <= end <= pay):
            return None
        count = min(chunk_elems, n - ci * chunk_elems)
        for k in range(0, count, 32):
            if pos + 4 > end:
                return None
            (mask,) = struct.unpack_from("<I", stream, base + pos)
            pos += 4
            valid = min(32, count - k)
            if mask >> valid:
                return None
            for i in range(valid):
                if mask >> i & 1:
                    if pos + 2 > end:
                        return None
                    out.append(struct.unpack_from("<H", stream, base + pos)[0])
                    pos += 2
                else:
                    out.append(0)
        if pos != end:
            return None
    return out

"""A short pure-Python fp64 restatement of one CSA decode query, written
separately from the C oracle, for brute-force pins on tiny inputs. Number
formats are decoded through torch's casts (a library routine)."""
import math
import struct

import torch

_E4M3 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).tolist()


def _bf16(b):
    return struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]


def _latent(rec, Dn, Dr, sb):
    rec = bytes(rec)
    scales = struct.unpack_from(f"<{(Dn + sb - 1) // sb}f", rec, Dn + 2 * Dr)
    rope = struct.unpack_from(f"<{Dr}H", rec, Dn)
    return [_E4M3[rec[d]] * scales[d // sb] for d in range(Dn)] + [_bf16(r) for r in rope]


def decode_one(qc, qs, w, kc, ks, p, m, N, k, q, sink, scale, comp, ring, W, Dn, Dr, sb):
    n_vis = min(p // m, N)
    logits = []
    for c in range(N):
        if c >= n_vis:
            logits.append(-math.inf)
            continue
        tot = 0.0
        for h in range(len(w)):
            dot = sum(_E4M3[qc[h][d]] * float(qs[h]) * _E4M3[kc[c][d]] * float(ks[c]) for d in range(len(kc[c])))
            tot += float(w[h]) * max(dot, 0.0)
        logits.append(tot)
    order = sorted(range(n_vis), key=lambda c: (-logits[c], c))
    sel = order[:min(k, n_vis)]
    cands = [_latent(comp[c], Dn, Dr, sb) for c in sel]
    cands += [_latent(ring[j % len(ring)], Dn, Dr, sb) for j in range(max(0, p - W + 1), p + 1)]
    outs, lses = [], []
    for h in range(len(q)):
        qh = [_bf16(v) for v in q[h]]
        z = [scale * sum(a * b for a, b in zip(qh, x)) for x in cands]
        M = max([float(sink[h])] + z)
        e = [math.exp(v - M) for v in z]
        den = math.exp(float(sink[h]) - M) + sum(e)
        outs.append([sum(e[j] * cands[j][d] for j in range(len(cands))) / den for d in range(Dn + Dr)])
        lses.append(M + math.log(den))
    return logits, sel, outs, lses

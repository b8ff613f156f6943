"""The 16-bit block format in which the two CTAs of a pair exchange partial logits
(test infrastructure, CPU): for each row and 64-key page, E = the exponent of the
largest |x_j| (its binade [2^E, 2^(E+1))), clamped to [-112, 127]; code
k_j = round-half-even(x_j * s) + 32768 with s = 2^(14-E) (1 - 2^-16) in fp32; the
receiver adds (k_j - 32768) * 2^(E-14) (1 + 2^-16).  Written from that definition in
numpy; it shares nothing with the kernel."""
import numpy as np


def block16_codes(x):
    """Codes and dequantised values of one block (a 1-D array of at most 64 fp32 values)."""
    x = np.asarray(x, dtype=np.float32)
    amax = float(np.abs(x).max()) if x.size else 0.0
    e = int(np.frexp(np.float32(amax))[1]) - 1 if amax > 0 else -127   # amax in [2^e, 2^(e+1))
    e = min(max(e, -112), 127)
    s = np.float32(2.0 ** (14 - e) * (1.0 - 2.0 ** -16))
    v = np.rint(x.astype(np.float64) * np.float64(s))     # the product is exact in float64
    k = v + 32768
    back = v * (2.0 ** (e - 14) * (1.0 + 2.0 ** -16))
    return k.astype(np.int64), back


def block16(x, block=64):
    """A row of partial logits as the receiving CTA sees it: blocks of `block` keys (pages)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    for j in range(0, len(x), block):
        out[j:j + block] = block16_codes(x[j:j + block].astype(np.float32))[1]
    return out

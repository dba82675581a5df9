"""Counter-based seeded bf16 inputs, evaluated on the host with numpy.

Every value is a pure function of (seed, rank, parameter, element index), so
any element of a 45 GB emulated gradient group can be regenerated on demand
without holding the group in host memory.  ``synth/csrc/synth_gen.cu``
implements the same definition on the GPU; the two must agree bit for bit.

Random bits: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014).  The generator's state
advances by the golden-ratio increment GAMMA and each output is the state
passed through the MIX64 finaliser; output i (0-based) of a stream seeded
with ``k`` is therefore ``mix64(k + (i + 1) * GAMMA)``, which is what makes
the generator counter-based.

Value maps (all integer arithmetic plus at most two fp32 multiplies, so the
host and the GPU round identically):

* UNIFORM   top 24 bits u -> (u - 2^23) * 2^-23 in [-1, 1), exact in fp32;
* NORMAL    Irwin-Hall sum of the four 16-bit fields of the 64-bit output,
            centred (|t| <= 131070, exact in fp32), times an fp32 scale that
            makes the standard deviation sigma -- an approximately normal
            N(0, sigma^2) with a hard tail at ~3.46 sigma;
* OUTLIER   NORMAL, then multiplied by 100 in fp32 when a second, independent
            SplitMix64 stream's top 24 bits fall below 0.1 * 2^24;
* INTEGER   (bits >> 32) mod 257 - 128, an integer in [-128, 128], exactly
            representable in bf16.

fp32 -> bf16 is round-to-nearest-even on the bit pattern (finite inputs only).
"""

import sys

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
OUTLIER_SALT = 0x5851F42D4C957F2D
_M64 = (1 << 64) - 1

UNIFORM = 0
NORMAL = 1
OUTLIER = 2
INTEGER = 3

# Irwin-Hall of four uniforms on {0..65535}: variance 4 * (65536^2 - 1) / 12.
IRWIN_HALL4_STD = float(np.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0))
OUTLIER_FACTOR = 100.0
OUTLIER_THRESHOLD = int(0.1 * (1 << 24))  # P(outlier) = 0.10


def mix64_int(z):
    """SplitMix64 finaliser on a Python int (reference form, used in tests)."""
    z &= _M64
    z = ((z ^ (z >> 30)) * MIX1) & _M64
    z = ((z ^ (z >> 27)) * MIX2) & _M64
    return z ^ (z >> 31)


def splitmix64_int(seed, i):
    """Output i (0-based) of the SplitMix64 stream seeded with ``seed``."""
    return mix64_int((seed + (i + 1) * GAMMA) & _M64)


def _mix64(z):
    """Vectorised SplitMix64 finaliser, in place on a uint64 array (wrapping)."""
    z ^= z >> np.uint64(30)
    z *= np.uint64(MIX1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(MIX2)
    z ^= z >> np.uint64(31)
    return z


def stream_bits(key, idx):
    """64 random bits for each element index in ``idx`` of stream ``key``."""
    z = np.array(idx, dtype=np.uint64, copy=True)
    z += np.uint64(1)
    z *= np.uint64(GAMMA)
    z += np.uint64(key)
    return _mix64(z)


def tensor_key(seed, rank, param):
    """Stream key of emulated rank ``rank``'s tensor ``param`` under ``seed``.

    The key is output number ``rank * 2^20 + param`` of the stream seeded with
    ``seed``; parameters are numbered below 2^20.
    """
    if not (0 <= param < (1 << 20)) or rank < 0:
        raise ValueError("rank must be >= 0 and param in [0, 2^20)")
    return splitmix64_int(seed, rank * (1 << 20) + param)


def normal_scale_f32(sigma):
    """fp32 scale that gives the Irwin-Hall sum a standard deviation ``sigma``.

    Computed once in fp64 and rounded to fp32 here; the GPU generator receives
    these exact fp32 bits rather than deriving them itself.
    """
    return np.float32(sigma / IRWIN_HALL4_STD)


def f32_to_bf16_bits(f):
    """Round finite fp32 values to bf16 (nearest, ties to even); uint16 bits."""
    b = np.asarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))
    return ((b + rounding) >> np.uint64(16)).astype(np.uint16)


def bf16_values(key, idx, dist, sigma=1e-3):
    """bf16 bit patterns (uint16) of stream ``key`` at element indices ``idx``."""
    bits = stream_bits(key, idx)
    if dist == UNIFORM:
        u = (bits >> np.uint64(40)).astype(np.int64) - (1 << 23)
        f = u.astype(np.float32) * np.float32(2.0 ** -23)
    elif dist in (NORMAL, OUTLIER):
        if sys.byteorder == "little":   # the four 16-bit fields, lowest first
            t = bits.view(np.uint16).reshape(-1, 4).sum(axis=1, dtype=np.int64)
        else:
            m16 = np.uint64(0xFFFF)
            t = ((bits & m16) + ((bits >> np.uint64(16)) & m16)
                 + ((bits >> np.uint64(32)) & m16) + (bits >> np.uint64(48))).astype(np.int64)
        t -= 2 * 65535
        f = t.astype(np.float32) * normal_scale_f32(sigma)
        if dist == OUTLIER:
            o = stream_bits(key ^ OUTLIER_SALT, idx) >> np.uint64(40)
            hit = o.astype(np.int64) < OUTLIER_THRESHOLD
            f = np.where(hit, f * np.float32(OUTLIER_FACTOR), f).astype(np.float32)
    elif dist == INTEGER:
        v = ((bits >> np.uint64(32)) % np.uint64(257)).astype(np.int64) - 128
        f = v.astype(np.float32)
    else:
        raise ValueError(f"unknown distribution {dist}")
    return f32_to_bf16_bits(f)


def bf16_tensor(key, numel, dist, sigma=1e-3, chunk=1 << 22):
    """A whole tensor of ``numel`` bf16 values (uint16 bits), built in chunks."""
    out = np.empty(numel, dtype=np.uint16)
    for a in range(0, numel, chunk):
        b = min(numel, a + chunk)
        out[a:b] = bf16_values(key, np.arange(a, b, dtype=np.uint64), dist, sigma)
    return out


def uniform01(key, idx):
    """Doubles in [0, 1) from the top 53 bits (used only to draw shapes)."""
    return (stream_bits(key, idx) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)

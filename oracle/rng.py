"""Counter-based random streams for the oracle (fp64, NumPy).

The write-ups only say that the rotation and the projection are "generated
mathematically" once and cached, never learned from data (Qiita TurboQuant
article, section "Rotate, then quantize"; DeepSignal TurboQuant article,
section "QJL"). They name no generator, so this project fixes one:

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014), counter form: draw k of stream ``seed`` is
  mix(seed + (k + 1) * golden_gamma);
* a uniform in [0, 1) from the top 53 bits; the first Box-Muller uniform is
  shifted to (0, 1] so its logarithm is finite;
* standard normals by Box-Muller, pair k taking draws 2k and 2k+1, cosine
  branch first.

The CUDA library's host code implements the same published definition on its
own; the two share no code.

Pinned by: the published SplitMix64 known-answer outputs for seed 0
(tests/golden/splitmix64_seed0.txt) and by distribution tests of the normals.
"""

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed, count, start=0):
    """Return draws ``start .. start+count-1`` of the SplitMix64 stream as uint64."""
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + k * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniforms(seed, count):
    """Uniforms in [0, 1): (draw >> 11) * 2**-53."""
    return (splitmix64(seed, count) >> np.uint64(11)).astype(np.float64) * 2.0**-53


def normals(seed, count):
    """``count`` standard normals by Box-Muller over the SplitMix64 stream."""
    pairs = (count + 1) // 2
    draws = splitmix64(seed, 2 * pairs).reshape(pairs, 2)
    u1 = ((draws[:, 0] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53
    u2 = (draws[:, 1] >> np.uint64(11)).astype(np.float64) * 2.0**-53
    rad = np.sqrt(-2.0 * np.log(u1))
    ang = 2.0 * np.pi * u2
    out = np.empty(2 * pairs, dtype=np.float64)
    out[0::2] = rad * np.cos(ang)
    out[1::2] = rad * np.sin(ang)
    return out[:count]


def sign_bits(seed, count):
    """±1 from the top bit of each draw: bit 63 set -> -1."""
    top = splitmix64(seed, count) >> np.uint64(63)
    return np.where(top == 1, -1.0, 1.0)


def round_to_bf16(x):
    """Round float64 values to the nearest bfloat16 (8 significant bits), ties to even.

    Direct from float64 (no float32 step, so no double rounding). Inputs are
    finite, inside the normal bfloat16 range, as the projection draws are.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)

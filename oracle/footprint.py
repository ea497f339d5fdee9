"""Cache footprint per token and KV head, fp64 oracle.

What the write-ups print: llama.cpp's turbo3 stores 3.25 bits per value at
about 4.9x less than FP16, turbo4 4.25 bits at about 3.8x (Qiita TurboQuant
article, "Which bit-width is 'lossless'", second table); with TQ3 a 70B model
on a 34 GB GPU goes from about 109K to about 536K tokens of context (Qiita,
"What you hit when you try it").

Reading: turbo3 / turbo4 correspond to keys in PROD mode at b = 3 / 4 bits
(b-1 Lloyd-Max bits + 1 QJL sign bit per coordinate) plus two float16 scalars
(n, gamma) per d = 128 coordinates.

Pinned by those printed figures (tests).
"""


def bytes_per_vector(mode, bits, d, m=None, padded=False, bits2=None):
    """Bytes one quantized vector occupies (codes + signs + float16 scalars);
    bits2: the second channel group's bits of a fractional rate (half the
    coordinates of every 16, see quantize.in_first_group)."""
    bprime = bits - 1 if mode == "prod" else bits
    code_bits = bprime * d
    if bits2 is not None:
        b2 = bits2 - 1 if mode == "prod" else bits2
        n1 = sum(1 for i in range(d) if i % 16 < 8)
        code_bits = bprime * n1 + b2 * (d - n1)
    code_bytes = (code_bits + 7) // 8
    if padded:
        code_bytes = (code_bytes + 15) // 16 * 16
    total = code_bytes + 2
    if mode == "prod":
        m = d if m is None else m
        sign_bytes = (m + 7) // 8
        if padded:
            sign_bytes = (sign_bytes + 15) // 16 * 16
        total += sign_bytes + 2
    return total


def bits_per_value(mode, bits, d, m=None, bits2=None):
    return 8.0 * bytes_per_vector(mode, bits, d, m, bits2=bits2) / d


def ratio_vs_fp16(mode, bits, d, m=None):
    return (2.0 * d) / bytes_per_vector(mode, bits, d, m)

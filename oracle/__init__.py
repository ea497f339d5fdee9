"""fp64 CPU oracle for TurboQuant online KV-cache quantization.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library, its
Python binding, the bench's GPU arm) imports, calls or links anything here.
Only the test suite, ``__graft_entry__.smoke()`` and the bench's
``cpu_baseline`` / ``--impl reference`` legs may use it.

Every function is a plain, slow restatement of what the method computes, in
float64 NumPy, following the steps in the order the write-ups describe them:

* rotation  - data-independent random orthogonal rotation (QR of a Gaussian
  matrix, or a random-sign Walsh-Hadamard transform);
* codebook  - Lloyd-Max scalar quantizer for the post-rotation coordinate law
  Beta((d-1)/2, (d-1)/2) on [-1, 1];
* quantize  - normalise, rotate, bucketize, bit-pack; for keys the 1-bit QJL
  sketch of the residual;
* attention - logits from the codes (pre-rotated query), exact softmax, value
  sum in the rotated domain, one un-rotation;
* topk      - inner-product search scored from the codes;
* polar     - the PolarQuant variant of the key quantizer (recursive polar
  transform of the rotated vector, one Lloyd-Max angle codebook per level).

It shares no code with the CUDA path; the two meet only through seeded inputs
built by ``online_kv_cache_quantize_gb300.workloads`` (which holds none of the
method's arithmetic) and through the packed-layout specification, which both
sides implement independently.

Parity status of each function is stated in its module docstring.
"""

from . import rng, rotation, codebook, quantize, attention, topk, footprint, polar  # noqa: F401

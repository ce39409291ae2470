"""Plain fp64 CPU oracle for TurboQuant's KV-cache quantizer and compressed-cache decode.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline / reference legs may import anything from this package.
The library (``kv_cache_vector_19_b300``) never imports it, and it imports nothing from
the library: the two share no code.  The only module both sides use is the seeded input
generator ``kv_cache_vector_19_b300.workloads``, which draws synthetic K/V/Q tensors and
contains none of the method's arithmetic.

Sources (web pages; each function cites the section it follows):

* [BLOG] "Технология TurboQuant и её применение с локальными LLM" (ast-softpro.ru blog),
  section 1.2 "Как работает TurboQuant": stage 1 = random orthogonal rotation followed
  by a per-coordinate MSE-optimal Lloyd-Max scalar quantizer with (b-1) bits; stage 2 =
  QJL: residual r = x - DEQUANT_mse(Q_mse(x)), projected by a random Gaussian matrix S,
  only sign(S r) stored, ||r||_2 kept as the reconstruction scale.
* [3BITS] "3 бита вместо 16: разбираем TurboQuant и когда его реально стоит включать"
  (kiosknews.app), section "Как работает TurboQuant": after the rotation the coordinates
  are nearly independent and close to normal; the Lloyd-Max codebook is computed once for
  that known distribution and stored statically, with no calibration (data-oblivious).
  Section "Python + HuggingFace": the quantizer returns (indices, norms) per vector.

Where the pages are silent the readings adopted are listed in each module's docstring.

Modules:
    rng       SplitMix64 counter stream and Box-Muller Gaussians (published definitions)
    rotation  Haar rotation Pi (QR of a Gaussian matrix, sign-fixed) and Gaussian S
    codebook  Lloyd-Max quantizer for one coordinate of a random unit vector in R^d
    quant     per-vector quantization of keys (MSE + QJL, or MSE only) and values (MSE)
    pagefmt   bit-exact packer / unpacker of the compressed page formats (version 1, and
              version 2 with separate key / value widths and optional QJL)
    decode    decode attention over the compressed cache (two equivalent routes)
"""

"""Oracle for the FibQuant codec: a plain, slow fp64 CPU statement of what the codec computes.

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the benchmark's CPU-baseline
leg may import this package. The library never calls it, and it never calls the library: the two
share no code. Its only inputs are the seeded draws of ``synth`` and caller-supplied arrays.

Citations ``[FibQuant §x]`` refer to section x of the page "FibQuant: universal vector quantisation
for random-access KV-cache compression" (gist.science summary of arXiv 2605.11478, Korean and
Dutch versions, which state the same content).

Parity status of each function (what pins it, in ``tests/test_oracle_*.py``):
  fibquant.row_norms           pinned (numpy.linalg.norm, closed forms)
  fibquant.rotate_normalise    pinned (unit norm invariant, Theorem 1 KS test, identity rotation)
  fibquant.nearest_codeword    pinned (scipy cKDTree exact NN, scalar midpoint rule, Q(c_n) = n)
  fibquant.pack / unpack       pinned (hand-worked golden bit vectors, round trip)
  fibquant.decode              pinned (equal-norm codebook round trip, identity rotation)
  codebook.haar_rotation       pinned (orthogonality, determinant, sign symmetry of the diagonal)
  codebook.companded_radii     pinned (k = 2 closed form against scipy betaincinv)
  codebook.spiral / kronecker  pinned (golden angle, Roberts constants as polynomial roots)
  codebook.lloyd               pinned (MSE non-increasing, MSE falls with N, beats scalar Lloyd-Max)
  fractal.vertices / encode    pinned (polygon closed forms, 40-digit unrolled recurrence)
  fractal.decode / access      pinned (exhaustive round trips, adversarial strings at the segment
                               limit, failure beyond it); fractal.append pinned against encode

The iterated-map archive (``fractal``) follows a second page, "Fractal KV-Cache Archives"
(gist.science summary of arXiv 2607.07144), cited there as [Archive §x].
"""

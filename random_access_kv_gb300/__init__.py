"""FibQuant KV-cache codec on GB300 (sm_103a): Python face of the C ABI in include/fq.h.

    ctx = fq_codebook_load(C, Pi)                    # shared codebook [N, k] and rotation [d, d]
    fq_encode(ctx, x, M, nu, codes)                  # x fp16 [M, d] -> nu fp32 [M], packed codes
    fq_decode_gather(ctx, nu, codes, M, idx, n, out) # random-access decode -> fp16 [n, d]

All device buffers are torch CUDA tensors owned by the caller; ``alloc_store`` sizes them.
``codebook`` builds the shared codebook and rotation on the host from seeded draws.
"""
from ._binding import (  # noqa: F401
    FQ_FLAG_NONFINITE, FQ_FLAG_RANGE, FQ_FLAG_TIMEOUT, Context, FQError, FQLibraryMissing,
    fq_attend, fq_centroid_sums, fq_code_words, fq_codebook_load, fq_decode, fq_decode_gather, fq_decode_gather_f32, fq_destroy,
    fq_encode, fq_encode_append, fq_record_bits, fq_selftest_wait, fq_shape, fq_status, fq_strerror, header_symbols,
)


def alloc_store(ctx, rows: int, device="cuda"):
    """Zeroed (nu fp32 [rows], codes int32 [fq_code_words(rows)]) torch tensors for a code store."""
    import torch
    nu = torch.zeros(rows, dtype=torch.float32, device=device)
    codes = torch.zeros(max(1, fq_code_words(ctx, rows)), dtype=torch.int32, device=device)
    return nu, codes

"""FibQuant KV-cache codec on GB300 (sm_103a): Python face of the C ABI in include/fq.h.

    ctx = fq_codebook_load(C, Pi)                    # shared codebook [N, k] and rotation [d, d]
    fq_encode(ctx, x, M, nu, codes)                  # x fp16 [M, d] -> nu fp32 [M], packed codes
    fq_decode_gather(ctx, nu, codes, M, idx, n, out) # random-access decode -> fp16 [n, d]

    actx = fa_create(N, r, L)                        # iterated-map archive of symbol streams
    fa_encode(actx, sym, n_streams, n_new, T_cap, T_old, anchors)   # append (T_old = 0: encode)
    fa_access(actx, anchors, n_streams, T_cap, T, pos, n, out)      # random access

All device buffers are torch CUDA tensors owned by the caller; ``alloc_store`` and
``alloc_archive`` size them.
``codebook`` builds the shared codebook and rotation on the host from seeded draws.
"""
from ._binding import (  # noqa: F401
    FQ_FLAG_NONFINITE, FQ_FLAG_RANGE, FQ_FLAG_TIMEOUT, Context, FQError, FQLibraryMissing,
    fq_attend, fq_centroid_sums, fq_code_words, fq_codebook_load, fq_decode, fq_decode_gather, fq_decode_gather_f32, fq_destroy,
    fq_encode, fq_encode_append, fq_record_bits, fq_selftest_wait, fq_shape, fq_status, fq_strerror, header_symbols,
    FA_FLAG_CORRUPT, FA_FLAG_RANGE, FA_FLAG_SYMBOL, ArchiveContext, fa_access, fa_create, fa_decode, fa_destroy,
    fa_encode, fa_max_segment, fa_params, fa_ratio_limit, fa_segments, fa_status, fa_vertex_table,
)


def alloc_store(ctx, rows: int, device="cuda"):
    """Zeroed (nu fp32 [rows], codes int32 [fq_code_words(rows)]) torch tensors for a code store."""
    import torch
    nu = torch.zeros(rows, dtype=torch.float32, device=device)
    codes = torch.zeros(max(1, fq_code_words(ctx, rows)), dtype=torch.int32, device=device)
    return nu, codes


def alloc_archive(ctx, n_streams: int, T_cap: int, device="cuda"):
    """Zeroed anchors float64 [n_streams, fa_segments(T_cap), 2] for an archive batch."""
    import torch
    return torch.zeros((n_streams, fa_segments(ctx, T_cap), 2), dtype=torch.float64, device=device)

/*
 * csa2.h -- C ABI of the CSA2 attention hot path on one GB300 (sm_103a).
 *
 * CSA2 (Compressed Sparse Attention 2) as described for DeepSeek-V4.1-Flash:
 *   hidden states -> non-overlapping compressor -> Main KV (FP4) -> Indexer K;
 *   Indexer Q x Indexer K -> score -> Top-K; Main Q attends to the selected Main KV
 *   plus the layer-local SWA KV.
 * Sources: "DeepSeek-V4.1-Flash deep dive" (tanjunchen.github.io, 2026-09-13),
 * sections 2, 3.1-3.4 and 6.3; "DeepSeek-V4.1-Flash paper reading" (inkeast, 2026-09-19)
 * section 4.2.
 *
 * Conventions shared by every call
 *   - Every pointer named "device" is a CUDA device pointer owned by the caller.  The
 *     library never allocates, frees or keeps device memory between calls (except one
 *     4-byte error word per device, see csa2_get_device_error, and the fixed score
 *     array of csa2_index_full_noalloc).
 *   - A call that takes a workspace (a device buffer of at least the bytes its *_workspace
 *     function reports, owned by the caller and free for the library's use until the
 *     call's work on the stream has completed) wants it 256-byte aligned: a misaligned
 *     workspace is rejected with CSA2_ERR_INVALID_ARG.
 *   - Every compute call is asynchronous on the given cudaStream_t (passed as void*;
 *     NULL = legacy default stream) and never synchronises.
 *   - Arguments are validated on the host before any launch; a failed check returns a
 *     status and csa2_last_error_message() (thread-local) says why.  Nothing is
 *     launched in that case.
 *   - Values that only the device can see (page ids read from a page table, n_vis,
 *     pool entries) are bounds-checked in the kernels: a bad value sets a bit in the
 *     device error word and the access is skipped (the row reads as zeros / the entry
 *     is ignored).  Kernels never trap.
 *   - Argument structs begin with struct_size = sizeof(struct) for ABI versioning.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *
 * Paged Main KV cache (one shared layout for the FP4 codes, the E4M3 scales and the
 * bf16 indexer K): entry e of sequence s lives on page page_table[s*max_pages + e/64],
 * slot e%64.  Each plane is an array of pages indexed by page id.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum csa2_status {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1,        /* NULL pointer, negative size, inconsistent sizes */
  CSA2_ERR_UNSUPPORTED_SHAPE = 2,  /* a size outside the supported set below */
  CSA2_ERR_WORKSPACE_TOO_SMALL = 3,
  CSA2_ERR_CUDA = 4,               /* a CUDA runtime call or launch failed */
  CSA2_ERR_DEVICE_CHECK = 5,       /* csa2_get_device_error: the word had a bounds-check bit */
  CSA2_ERR_TIMEOUT = 6             /* csa2_get_device_error: the word had CSA2_DEVERR_TIMEOUT */
} csa2_status;

/* Element types.  CSA2_FP8E4M3 selects the compressed indexer-K plane (csa2_cache);
 * CSA2_FP4E2M1X2 names the packed Main KV codes (two E2M1 codes per byte), which no
 * argument takes as a choice. */
typedef enum csa2_dtype { CSA2_BF16 = 0, CSA2_F32 = 1, CSA2_FP8E4M3 = 2, CSA2_FP4E2M1X2 = 3 } csa2_dtype;

/* Device error word bits (csa2_get_device_error). */
#define CSA2_DEVERR_PAGE_ID      0x1u  /* page id outside [0, num_pages) */
#define CSA2_DEVERR_PAGE_SLOT    0x2u  /* entry index beyond max_pages*page_size */
#define CSA2_DEVERR_N_VIS        0x4u  /* n_vis[b] outside [0, max_n] */
#define CSA2_DEVERR_POOL_ENTRY   0x8u  /* pool_len[b] out of range */
#define CSA2_DEVERR_SEQ          0x10u /* seq_of / seq index outside [0, num_seqs) */
#define CSA2_DEVERR_SWA_RANGE    0x20u /* SWA window outside [0, swa_rows) */
#define CSA2_DEVERR_POS          0x40u /* RoPE position outside [0, rope_max_pos) */
#define CSA2_DEVERR_TIMEOUT      0x80u /* a bounded wait on tensor-core or TMA completion gave up */
#define CSA2_DEVERR_SMEM_ALIGN   0x100u /* dynamic shared memory was not 1024-byte aligned */

#define CSA2_PAGE_SIZE 64

/* Paged cache planes (all device).  d in {128, 512}; d_ik in {64, 128};
 * num_pages <= 2^25 (2^31 entries).
 *
 * Indexer K is kept in one of two forms, chosen by idx_k_dtype:
 *   CSA2_BF16    (0, the form the pages imply): idx_k, bf16.
 *   CSA2_FP8E4M3 (compressed; not on the pages): idx_k8 and idx_k8_scale -- each entry's
 *                bf16 indexer K row x quantised to E4M3 with one float32 scale:
 *                s = amax|x| / 448 (float32 division), byte = E4M3_RNE_satfinite(x / s),
 *                s == 0 -> zero bytes (the quantiser of csa2_swa_quant).  d_ik + 4 bytes
 *                an entry instead of 2 d_ik: the Full scan streams half the bytes.  The
 *                indexer then quantises each query head's bf16 indexer Q the same way and
 *                scores the dequantised values:
 *                s(e) = sum_h w_h ReLU((sq_h q8_h) . (sk_e k8_e)),
 *                its dot products on FP8 tensor-core operands (exact products, float32
 *                sums).
 */
typedef struct csa2_cache {
  uint8_t* codes;              /* [num_pages][64][d/2]  E2M1 pairs, even channel in the low nibble;
                                  16-byte aligned */
  uint8_t* scales;             /* [num_pages][64][d/16] E4M3 scale of each 16 channels; 16-byte aligned */
  uint16_t* idx_k;             /* [num_pages][64][d_ik] bf16 indexer K (CSA2_BF16 form; may be NULL
                                  if unused); 16-byte aligned */
  const int32_t* page_table;   /* [num_seqs][max_pages] page id of each 64-entry page */
  int32_t num_pages;
  int32_t page_size;           /* must be 64 */
  int32_t num_seqs;
  int32_t max_pages;
  int32_t d;
  int32_t d_ik;
  csa2_dtype idx_k_dtype;      /* CSA2_BF16 (0) or CSA2_FP8E4M3 */
  uint8_t* idx_k8;             /* [num_pages][64][d_ik] E4M3 indexer K (CSA2_FP8E4M3 form); 16-byte
                                  aligned */
  float* idx_k8_scale;         /* [num_pages][64] float32 scale of each idx_k8 row; 16-byte aligned */
} csa2_cache;

/* ------------------------------------------------------------------------------
 * csa2_compress_quant -- the non-overlapping compressor and FP4 quantiser.
 * deep dive section 2: C = H.W_KV, Z = H.W_Z; section 3.1: every m tokens become one
 * Main KV entry (no overlap, no absolute PE) and Indexer K is projected from Main KV;
 * section 3.4: RoPE, then FP4 E2M1 with one E4M3 scale per 16 channels.
 *
 * For each group g of m consecutive input rows [g*m, g*m+m):
 *   e[c]  = sum_j softmax_j(Z[g*m+j][c]) * C[g*m+j][c]        (float32)
 *   y     = RoPE(e) on the last d_rope channels: pair i = channels
 *           (d-d_rope+2i, d-d_rope+2i+1), angle from rope_cos/rope_sin[pos[g]][i],
 *           y0 = x0*c - x1*s, y1 = x0*s + x1*c, each product rounded (no FMA)
 *   per 16 channels: s = E4M3_RNE_satfinite(amax/6); codes = E2M1_RNE_sat(y/s)
 *           (float32 divisions, correctly rounded; s == 0 gives zero codes)
 *   idx_k = bf16_RNE(dequant(codes, s) . W_ik)                  (if W_ik != NULL)
 * and writes entry entry[g] of sequence seq[g] through the page table.
 *
 * Modes:
 *   projection: W_kv != NULL.  H is [T][d_model] (h_dtype bf16 or f32), W_kv and W_z
 *               are bf16 [d_model][d] (W_z may be NULL when m == 1).  C and Z are
 *               computed in float32 into the workspace.
 *   given:      W_kv == NULL.  C (and Z when m > 1) are float32 [T][d] device arrays.
 * Supported: m in 1..8, d in {128, 512}, d_ik in {64, 128}, d_rope in {0, 32, 64},
 * d_rope <= d, d_model % 32 == 0, T % m == 0.
 * -------------------------------------------------------------------------- */
typedef struct csa2_compress_args {
  size_t struct_size;
  int32_t T;                   /* input rows */
  int32_t m;                   /* compression ratio */
  int32_t d_model;             /* projection mode only */
  csa2_dtype h_dtype;          /* projection mode only */
  const void* H;               /* device [T][d_model] */
  const uint16_t* W_kv;        /* device bf16 [d_model][d], NULL = given mode */
  const uint16_t* W_z;         /* device bf16 [d_model][d] */
  const float* C;              /* device f32 [T][d] (given mode) */
  const float* Z;              /* device f32 [T][d] (given mode, m > 1) */
  int32_t d_rope;              /* 0 disables RoPE */
  int32_t rope_max_pos;        /* rows of the tables */
  const float* rope_cos;       /* device f32 [rope_max_pos][d_rope/2] */
  const float* rope_sin;       /* device f32 [rope_max_pos][d_rope/2] */
  const int32_t* pos;          /* device [T/m] RoPE position of each group */
  const int32_t* seq;          /* device [T/m] destination sequence of each group */
  const int32_t* entry;        /* device [T/m] destination entry index of each group */
  const uint16_t* W_ik;        /* device bf16 [d][d_ik], NULL = do not write idx_k */
  csa2_cache cache;            /* destination planes */
  float* y_out;                /* device f32 [T/m][d] pre-quantisation rows, or NULL */
} csa2_compress_args;

csa2_status csa2_compress_quant(const csa2_compress_args* args, void* workspace,
                                size_t workspace_bytes, void* stream);
csa2_status csa2_compress_quant_workspace(const csa2_compress_args* args, size_t* bytes);

/* ------------------------------------------------------------------------------
 * csa2_compress_append -- the decode-time cache append: one new token for each of B
 * sequences, at compression ratio m (deep dive 3.1: every m tokens become one Main KV
 * entry -- the encoder's m = 2, the decoder's m = 1).
 *
 * An entry exists once all m of its tokens exist, so a token that does not complete its
 * group waits: for the token at position t = tok_pos[b] of sequence s = seq[b],
 *   C = H[b].W_kv and Z = H[b].W_z (float32) are stored as row t % m of the sequence's
 *   pending group pend[s] (C rows [m][d], then Z rows [m][d]);
 *   if t % m == m - 1 the group is complete: its m rows are pooled, rotated at position t
 *   and quantised exactly as csa2_compress_quant does for m consecutive rows, written as
 *   entry t / m of sequence s, and its indexer K projected (when W_ik != NULL).
 * pend holds each sequence's waiting tokens between calls; the caller keeps it (no
 * initialisation is needed: a group's rows are written before they are read, as long as
 * every sequence's tokens are appended in order).  At m = 1 pend is not used.  The tokens
 * of one call must belong to distinct sequences.  y_out (optional, [B][d] float32)
 * receives the pre-quantisation row of each token that completes a group; the rows of
 * the other tokens are left unchanged.
 * Device checks: seq outside [0, cache.num_seqs) sets CSA2_DEVERR_SEQ, a negative tok_pos
 * CSA2_DEVERR_POS, and that token is skipped.
 * Supported: as csa2_compress_quant's projection mode (m in 1..8, d in {128, 512},
 * d_model % 32 == 0, bf16 or f32 H).
 * -------------------------------------------------------------------------- */
typedef struct csa2_append_args {
  size_t struct_size;
  int32_t B;                   /* new tokens, each of a different sequence */
  int32_t m;                   /* compression ratio */
  int32_t d_model;
  csa2_dtype h_dtype;
  const void* H;               /* device [B][d_model] hidden state of each new token */
  const uint16_t* W_kv;        /* device bf16 [d_model][d] */
  const uint16_t* W_z;         /* device bf16 [d_model][d], required when m > 1 */
  int32_t d_rope;              /* 0 disables RoPE */
  int32_t rope_max_pos;
  const float* rope_cos;       /* device f32 [rope_max_pos][d_rope/2] */
  const float* rope_sin;
  const int32_t* seq;          /* device [B] sequence of each token */
  const int32_t* tok_pos;      /* device [B] position of each token in its sequence */
  float* pend;                 /* device f32 [cache.num_seqs][2][m][d] (m > 1; NULL at m = 1) */
  const uint16_t* W_ik;        /* device bf16 [d][d_ik], NULL = do not write idx_k */
  csa2_cache cache;            /* destination planes */
  float* y_out;                /* device f32 [B][d] or NULL */
} csa2_append_args;

csa2_status csa2_compress_append(const csa2_append_args* args, void* workspace, size_t workspace_bytes,
                                 void* stream);
csa2_status csa2_compress_append_workspace(const csa2_append_args* args, size_t* bytes);

/* ------------------------------------------------------------------------------
 * csa2_index_full -- Full-mode hierarchical sparse indexer.
 * deep dive 3.3: the first Full indexer scans the whole causally visible range, keeps
 * the best positions of each block; 2,048 blocks x 8 = a 16,384-candidate shared pool;
 * Top-512 per query.  deep dive 3.1: Indexer Q x Indexer K -> score -> Top-K.
 *
 * For query b over the visible entries [0, n = n_vis[b]) of sequence seq_of[b]:
 *   s(e)  = sum_h w[b][h] * ReLU(q_idx[b][h] . idx_k[e])   (relu = 0: no ReLU)
 *   block j = [floor(j*n/NB), floor((j+1)*n/NB)), keep the best min(per_block, len),
 *   pool  = union of the kept entries, ascending; pool_len = min(n, NB*per_block);
 *   topk  = best min(k, pool_len) entries of the pool, ascending.
 * "Best" = larger score; equal scores go to the lower entry index.
 * Outputs (device): pool [B][NB*per_block] and topk [B][k], -1 padded; pool_len,
 * topk_len [B].  Scores are float32 on the device.
 * Supported: H_i in 1..32, d_ik in {64, 128}, per_block in 1..32, NB*per_block <= 16384,
 * k in 1..2048, max_n <= max_pages*64.
 *
 * group (0 or 1: every query alone): queries g*group .. g*group+group-1 belong to one
 * sequence (equal seq_of; a mismatch sets CSA2_DEVERR_SEQ); n_vis may differ within a group;
 * needs B % group == 0.  Each indexer-K row is then read once for the whole group -- e.g. the
 * 1 + 5 positions of a speculative-decoding verification step, or the causal queries of a
 * prefill chunk.
 * Tensor-core scoring: with H_i in {8, 16, 32}, d_ik = 128, per_block <= 16 and 16-byte
 * aligned q_idx, w and idx_k, the scores are one tcgen05 product of a group's indexer Q
 * (group x H_i columns, at most 256; a larger group must be a multiple of 256 / H_i)
 * against the cache's indexer K, float32 accumulation, written to the workspace (B * max_n
 * floats more), after which each block keeps its best.  It is taken whenever group x H_i >=
 * 16 (so also by single queries with 16 or 32 heads); a single 8-head query keeps the
 * scan.  The accumulation order differs from the scan's, so near-ties may resolve
 * differently.  Otherwise groups of 2..8 queries with H_i <= 8 are scanned together (the
 * results of scanning every query alone), and other groups query by query.
 * csa2_index_full_noalloc never takes the tensor-core scoring.
 * -------------------------------------------------------------------------- */
typedef struct csa2_index_full_args {
  size_t struct_size;
  int32_t B;
  int32_t H_i;
  const uint16_t* q_idx;       /* device bf16 [B][H_i][d_ik] */
  const float* w;              /* device f32 [B][H_i] */
  csa2_cache cache;            /* idx_k + page_table */
  const int32_t* seq_of;       /* device [B] */
  const int32_t* n_vis;        /* device [B] visible entries per query */
  int32_t max_n;               /* host bound: every n_vis[b] <= max_n */
  int32_t num_blocks;          /* NB */
  int32_t per_block;
  int32_t k;
  int32_t relu;
  int32_t* pool;               /* device [B][NB*per_block] */
  int32_t* pool_len;           /* device [B] */
  int32_t* topk;               /* device [B][k] */
  int32_t* topk_len;           /* device [B] */
  int32_t group;               /* queries scanned together (see above); 0 = 1 */
} csa2_index_full_args;

csa2_status csa2_index_full(const csa2_index_full_args* args, void* workspace,
                            size_t workspace_bytes, void* stream);
csa2_status csa2_index_full_workspace(const csa2_index_full_args* args, size_t* bytes);

/* ------------------------------------------------------------------------------
 * csa2_index_full_noalloc -- csa2_index_full for callers that cannot allocate device
 * memory.  The pages have no counterpart to this call: it is a convenience of the
 * library, not a step of the method.
 *
 * Some callers cannot hand the library a workspace: a serving process that carved all
 * of HBM into KV pages at start-up and has no allocator left, a host runtime that talks
 * to the library through this C ABI without any CUDA allocator of its own, or code
 * that must not call cudaMalloc on its hot path (an allocation can synchronise the
 * device and stall every stream).  This entry point needs no workspace: the candidate
 * scores it needs between its two kernels live in one fixed device array compiled into
 * the library, CSA2_NOALLOC_MAX_SCORES floats (4 MiB).  Every GPU that loads the
 * library holds that array until the process exits.  The call itself allocates nothing.
 *
 * Arguments and outputs are those of csa2_index_full, and so are the results whenever
 * csa2_index_full scans (group x H_i < 16, or a shape the tensor-core scoring does not
 * take): this call always scans, because the fixed array holds the pool scores only, not
 * the tensor-core score matrix.  Where csa2_index_full scores on the tensor cores instead
 * (group x H_i >= 16 with H_i in {8, 16, 32}, see above), the two calls accumulate the
 * float32 scores in different orders, so an entry whose score ties another's to within
 * rounding may be kept by one call and not the other; both results satisfy the same
 * near-tie rule against the exact scores.  Limits and rules of the shared array:
 *   - B * num_blocks * per_block must not exceed CSA2_NOALLOC_MAX_SCORES (with the
 *     16,384-candidate pool that is B <= 64); larger calls return
 *     CSA2_ERR_UNSUPPORTED_SHAPE and launch nothing.
 *   - The array's device address belongs to a CUDA context.  The first call in a context
 *     (the device's primary one, another one made current, or a new one after
 *     cudaDeviceReset) looks it up with the device current; make that first call before
 *     any stream capture.
 *   - All calls on a device share the one array and it keeps the previous call's
 *     contents.  Nothing in it needs to start at zero (every score is written before it
 *     is read), but calls that overlap on the GPU -- on two streams, or from two host
 *     threads -- race on it and must be serialised by the caller.
 * -------------------------------------------------------------------------- */
#define CSA2_NOALLOC_MAX_SCORES (1 << 20)

csa2_status csa2_index_full_noalloc(const csa2_index_full_args* args, void* stream);

/* ------------------------------------------------------------------------------
 * csa2_index_reindex -- Reindex mode (deep dive 3.2, 3.3 step 3): this layer's own
 * indexer Q re-scores only the shared pool (entries of the cache built by the Full
 * layer) and picks its own Top-k.  Same score and ordering rules as csa2_index_full.
 * pool: [B][pool_stride] ascending entry indices, the first pool_len[b] valid.
 * Reuse mode (deep dive 3.2) needs no call: pass the previous topk to csa2_sparse_attn.
 * -------------------------------------------------------------------------- */
typedef struct csa2_index_reindex_args {
  size_t struct_size;
  int32_t B;
  int32_t H_i;
  const uint16_t* q_idx;       /* device bf16 [B][H_i][d_ik] */
  const float* w;              /* device f32 [B][H_i] */
  csa2_cache cache;
  const int32_t* seq_of;       /* device [B] */
  const int32_t* pool;         /* device [B][pool_stride] */
  const int32_t* pool_len;     /* device [B] */
  int32_t pool_stride;         /* <= 16384 */
  int32_t k;
  int32_t relu;
  int32_t* topk;               /* device [B][k] */
  int32_t* topk_len;           /* device [B] */
} csa2_index_reindex_args;

csa2_status csa2_index_reindex(const csa2_index_reindex_args* args, void* workspace,
                               size_t workspace_bytes, void* stream);
csa2_status csa2_index_reindex_workspace(const csa2_index_reindex_args* args, size_t* bytes);

/* ------------------------------------------------------------------------------
 * csa2_sparse_attn -- one softmax over the selected FP4 Main KV entries plus the
 * layer-local FP8 SWA window (deep dive 3.1; 6.3: 64 query heads x 512, n_win 128,
 * Top-K 512).  The entry vector is both key and value (MQA over the shared entry).
 *
 * For query b and head h, S = { topk[b][i] : i < topk_len[b], topk[b][i] >= 0 }
 *   U { SWA rows swa_start[b] .. swa_start[b]+swa_len[b]-1 }:
 *   l_s = softmax_scale * q[b][h] . kv_s;  p = softmax_S(l);  out[b][h] = sum_s p_s kv_s
 *   kv_s = dequant FP4 entry (exact) or E4M3 row * swa_scale[row].
 *   lse[b][h] = log(sum_s exp(l_s)) (natural log); empty S gives out = 0, lse = -inf.
 * Precision: the products run on fp16 tensor-core operands with float32 accumulation.
 * The keys are exact there (the dequantised FP4 entries and the window rows' E4M3 values);
 * a window row's scale is applied in float32 to its logit and to its weight in P.V; each
 * head's q is scaled by a power of two before its fp16 rounding (exact for every bf16
 * element within 2^-28 of the head's largest), and the probabilities are fp16 (2^-12
 * relative).  Inputs: any finite bf16 q, any E4M3 scale byte but the NaN patterns 0x7F /
 * 0xFF, any finite swa_scale; the logits softmax_scale * q . kv must be finite in float32.
 * Supported: Hq in {8, 16, 32, 64}, d in {128, 512}, k + swa_max <= 4096.
 * -------------------------------------------------------------------------- */
typedef struct csa2_attn_args {
  size_t struct_size;
  int32_t B;
  int32_t Hq;
  const uint16_t* q;           /* device bf16 [B][Hq][d] */
  csa2_cache cache;            /* codes, scales, page_table, d */
  const int32_t* seq_of;       /* device [B] */
  const int32_t* topk;         /* device [B][k] */
  const int32_t* topk_len;     /* device [B], or NULL = all k slots */
  int32_t k;
  const uint8_t* swa;          /* device E4M3 [swa_rows][d] (may be NULL if swa_max == 0) */
  const float* swa_scale;      /* device f32 [swa_rows] */
  int32_t swa_rows;
  const int32_t* swa_start;    /* device [B] */
  const int32_t* swa_len;      /* device [B] */
  int32_t swa_max;             /* host bound: every swa_len[b] <= swa_max */
  float softmax_scale;
  void* out;                   /* device [B][Hq][d] */
  csa2_dtype out_dtype;
  float* lse;                  /* device f32 [B][Hq], or NULL */
  int32_t inputs_ready;        /* 1: none of this call's inputs (q, topk, topk_len, seq_of, the
                                  cache, the window rows and scales) is written by a kernel launched
                                  on the stream since the last library call made without this flag
                                  -- e.g. a Reuse layer's attention after the attention calls of the
                                  layers since the last index call, which write only their own
                                  outputs.  The call then reads and computes while those kernels
                                  finish, and waits for them only before its first write (so its
                                  writes stay in stream order).  0: it waits before its first
                                  read, as every other call does. */
} csa2_attn_args;

csa2_status csa2_sparse_attn(const csa2_attn_args* args, void* workspace,
                             size_t workspace_bytes, void* stream);
csa2_status csa2_sparse_attn_workspace(const csa2_attn_args* args, size_t* bytes);

/* ------------------------------------------------------------------------------
 * csa2_swa_quant -- FP8 window rows with one float32 scale per row: the step that
 * rebuilds a layer's SWA window when its last tokens are replayed (deep dive 3.4, "SWA
 * Bounded Replay": SWA KV stays FP8; the replayed tokens' window is recomputed rather
 * than kept).  The replayed rows themselves (the layer's projections of those tokens'
 * hidden states) are inputs.  For each input row r:
 *   a = max_i |x[r][i]|;  s = a / 448 (float32 division, correctly rounded);
 *   s == 0 -> every byte 0;  else byte_i = E4M3_RNE_satfinite(x[r][i] / s)  (float32
 *   division);  swa[dst][i] = byte_i, swa_scale[dst] = s,  dst = row_idx[r] (or r).
 * csa2_sparse_attn then attends over the rebuilt window (k = 0 for the window alone).
 * A dst outside [0, swa_rows) sets CSA2_DEVERR_SWA_RANGE and that row is skipped.
 * Supported: d in {128, 512}; x bf16 or f32, 16-byte aligned; swa 16-byte aligned
 * (d = 512) or 4-byte aligned (d = 128).  Needs no workspace.
 * -------------------------------------------------------------------------- */
typedef struct csa2_swa_quant_args {
  size_t struct_size;
  int32_t R;                   /* rows to quantise */
  int32_t d;                   /* row width */
  csa2_dtype x_dtype;          /* CSA2_BF16 or CSA2_F32 */
  const void* x;               /* device [R][d] */
  const int32_t* row_idx;      /* device [R] destination row of each input row, or NULL = r */
  uint8_t* swa;                /* device E4M3 [swa_rows][d] */
  float* swa_scale;            /* device f32 [swa_rows] */
  int32_t swa_rows;
} csa2_swa_quant_args;

csa2_status csa2_swa_quant(const csa2_swa_quant_args* args, void* stream);

/* ------------------------------------------------------------------------------
 * Helpers
 * -------------------------------------------------------------------------- */

/* Thread-local description of the last failed call ("" if none). */
const char* csa2_last_error_message(void);

/* Synchronises the current device, stores the device error word (CSA2_DEVERR_* bits)
 * accumulated since the last read in *word, and clears it.  Returns CSA2_OK for a zero
 * word, CSA2_ERR_TIMEOUT when the word has CSA2_DEVERR_TIMEOUT, CSA2_ERR_DEVICE_CHECK
 * when it has any other bit (CSA2_ERR_CUDA if the synchronisation failed; *word is then
 * not written).  For tests and debugging: it blocks.  The word is per device, not per
 * stream, so the call takes no stream. */
csa2_status csa2_get_device_error(uint32_t* word);

/* Library version: major*10000 + minor*100 + patch. */
int32_t csa2_version(void);

/* ------------------------------------------------------------------------------
 * csa2_selftest_wait_timeout -- exercises the failure path of the library's bounded
 * waits.  Every wait of the tensor-core kernels (on an mbarrier or a cluster peer)
 * gives up after a fixed number of polls, sets CSA2_DEVERR_TIMEOUT in the device error
 * word, skips the work that depended on it and returns, so the context stays usable.
 * This call launches one CTA that waits on an mbarrier that nothing arrives on, giving
 * up after `polls` polls (1 <= polls <= 2^20), so that path can be tested without a
 * fault.  It touches no memory outside the CTA.  The pages have no counterpart to it.
 * -------------------------------------------------------------------------- */
csa2_status csa2_selftest_wait_timeout(int32_t polls, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H */

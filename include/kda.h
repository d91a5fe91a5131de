/*
 * kda.h -- C ABI of the GB300 (sm_103a) KDA speculative verify / commit
 * library ("RecoverSSM": one checkpoint state per request).
 *
 * The pages this follows:
 *   [GLM]  recipes/docker-images/glm53-kindling/experimental/fixes/recoverssm.py
 *          (GLM-5.3-Flash KDA speculative verify with one checkpoint state per
 *          request): `_verify_kernel`, `kda_recoverssm_verify`,
 *          `_prepare_commit_plan_kernel`, `Glm5NextRecoverSSMCommitContext.commit`.
 *   [KIMI] vllm.models.kimi_k3.nvidia.specialized_decode.recoverssm.context
 *          (the deferred fp32 commit): `KDADeferredCommitContext.commit`,
 *          `.flush`, `KDARecoverSSMDeferred`, `allocate_records`.
 *   [LAYER] recipes/.../experimental/fixes/kda.py (GLM-5.3-Flash KDA layer):
 *          the gate (bounded sigmoid or the default softplus) and the layout
 *          of q, k, v, g_raw and beta_raw.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *   never allocates, never synchronises the stream and never reads device
 *   data on the host, so every call is a pure stream-ordered launch.
 * - Sizes: K = V = head_dim = 128; Q = window = 1 + num_spec, 1..8.
 * - The recurrent state pool is fp32 [num_slots][H][V][K], K contiguous, one
 *   64 KiB tile per (slot, head).  Slot 0 is the null block: rows whose state
 *   index is <= 0 are padding and are skipped entirely ([GLM] verify kernel).
 * - Activations are bf16.  q, k, v, g_raw: [T_total][H][128] with a token
 *   stride given in elements (heads contiguous inside a token); beta_raw:
 *   [T_total][H] with its own token stride.  cu_seqlens is int32 [B + 1]
 *   (row b owns tokens cu_seqlens[b] .. cu_seqlens[b+1]-1).
 * - Records (the verify -> commit scratch of [GLM] `Records` and [KIMI]
 *   `allocate_records`) hold each token's RAW bf16 k, v, g_raw and beta_raw
 *   (or, with cfg->record_format == KDA_RECORDS_CORRECTION, its fp32 delta
 *   with k and g_raw; see KDA_RECORDS_CORRECTION below).
 *   They are indexed by record slot r in [-1, R): r = -1 is a scratch row
 *   that rows without a record slot write and nothing ever reads.  Raw
 *   layout (internal, sized by kda_records_bytes): bf16
 *   [R + 1][H][Q][KDA_RECORD_STRIDE] with record slot r at row r + 1, and in
 *   each token record k at [0,128), v at [128,256), g_raw at [256,384) and
 *   beta_raw at element 384 (the rest is padding to a 16-byte multiple).
 * - record_rows: int32 [B], the record slot of each row, or NULL for r = b
 *   (the GLM per-row layout, which then requires B <= R).
 * - pending: int32 [R], per record slot, the accepted count whose replay is
 *   still to be folded ([KIMI] `KDARecoverSSMDeferred.pending`).
 * - error_word: optional device int32; a kernel that meets bad metadata skips
 *   the row and ORs a KDA_ROW_* bit into it (no trap, no abort).  NULL: the
 *   bits are dropped.
 * - stream: a cudaStream_t passed as void* (NULL: the legacy default stream).
 * - Return value: KDA_OK after a successful launch (or when there is nothing
 *   to launch, e.g. B == 0); KDA_ERR_INVALID_ARG / KDA_ERR_UNSUPPORTED when a
 *   host-side check fails (nothing is launched); KDA_ERR_CUDA when the launch
 *   itself fails (cudaGetLastError after the launch).
 * - Rows must use distinct state slots and distinct record slots (other than
 *   -1); two rows sharing one race, as in the pages.
 */
#ifndef KDA_GB300_KDA_H
#define KDA_GB300_KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* a pointer, size, stride, alignment or format is wrong */
    KDA_ERR_UNSUPPORTED = 2,  /* valid but not built: head_dim != 128, Q > 8, H > 32767 */
    KDA_ERR_CUDA = 3          /* the kernel launch failed */
} kda_status;

/* Bits of *error_word (device-side checks; the row is skipped). */
#define KDA_ROW_BAD_LENGTH  1  /* token count < 0 or > window */
#define KDA_ROW_BAD_SLOT    2  /* state index >= num_slots */
#define KDA_ROW_BAD_RECORD  4  /* record slot outside [-1, record_slots) */
#define KDA_ROW_BAD_PENDING 8  /* pending count outside [0, window] */
/* A kernel gave up waiting (about 2 s) for one of its own asynchronous copies
 * into shared memory and returned early; its remaining rows were not
 * processed.  Not expected in normal operation. */
#define KDA_ERR_WAIT_TIMEOUT 16
/* align mode: request index outside the block table, negative num_computed,
 * or a boundary block past the table's last column */
#define KDA_ROW_BAD_BLOCK 32

#define KDA_HEAD_DIM 128
#define KDA_MAX_WINDOW 8
#define KDA_MAX_HEADS 32767
/* elements (bf16) per token record: k, v, g_raw (3 x 128), beta_raw, padding */
#define KDA_RECORD_STRIDE 392

/* Record formats (kda_config.record_format).
 * KDA_RECORDS_RAW: each token's raw bf16 k, v, g_raw and beta_raw; a commit,
 *   fold or flush replays the recurrence on them ([GLM] `Records`).
 * KDA_RECORDS_CORRECTION: each token's fp32 delta v' = beta (v - S k^) (the
 *   "correction" of [KIMI] `allocate_records`, whose fp32 [Q, D] and
 *   activation-dtype [Q, 2D] tensors these mirror) with its bf16 k and g_raw;
 *   a commit, fold or flush applies S <- S diag(exp(g)) + v' k^T per token,
 *   i.e. folds the deltas in closed form, without the prediction S k^.
 *   Layout (internal, sized by kda_correction_records_bytes): per record slot
 *   row r + 1, head h and token t, KDA_CORRECTION_RECORD_BYTES bytes: the
 *   fp32 delta of the 128 rows at byte 0, bf16 k at byte 512, bf16 g_raw at
 *   byte 768.  The folded state has the bits of the verify's trajectory (the
 *   same operations in the same order after v'), as in the raw format. */
#define KDA_RECORDS_RAW 0
#define KDA_RECORDS_CORRECTION 1
#define KDA_CORRECTION_RECORD_BYTES 1024

typedef struct kda_config {
    int32_t num_heads;        /* 1 <= H <= KDA_MAX_HEADS */
    int32_t head_dim;         /* must be 128 (K = V) */
    int32_t window;           /* Q = 1 + num_spec, 1..8 */
    int32_t num_slots;        /* S: slots of the state pool (slot 0 = null) */
    int32_t record_slots;     /* R: record slots (the scratch row excluded) */
    int32_t use_lower_bound;  /* 1: bounded sigmoid gate, 0: softplus gate */
    float lower_bound;        /* < 0, used when use_lower_bound == 1 */
    float scale;              /* multiplies the normalised q (head_dim^-0.5) */
    int64_t stride_q_t;       /* token strides in elements; q, k, v and g_raw */
    int64_t stride_k_t;       /*   need multiples of 4 and 8-byte aligned bases */
    int64_t stride_v_t;
    int64_t stride_g_t;
    int64_t stride_beta_t;    /* any positive stride */
    int32_t record_format;    /* KDA_RECORDS_RAW or KDA_RECORDS_CORRECTION; every
                                 call on one records buffer must use the same */
    int32_t reserved;         /* must be 0 */
} kda_config;

/* Bytes of the raw-format records buffer for H heads, window Q and R record
 * slots: (R + 1) * H * Q * KDA_RECORD_STRIDE * 2.  0 for invalid sizes. */
size_t kda_records_bytes(int32_t num_heads, int32_t window, int32_t record_slots);

/* Bytes of a correction-format records buffer:
 * (R + 1) * H * Q * KDA_CORRECTION_RECORD_BYTES.  0 for invalid sizes. */
size_t kda_correction_records_bytes(int32_t num_heads, int32_t window, int32_t record_slots);

/*
 * kda_verify -- speculative verify from each row's checkpoint
 * ([GLM] `_verify_kernel` / `kda_recoverssm_verify`).
 *
 * For each row b with T = cu_seqlens[b+1] - cu_seqlens[b] tokens and state
 * slot s = state_indices[b] > 0, and each head h, starting from the fp32
 * tile state_pool[s][h]:
 *   per token: q^ = q/sqrt(|q|^2+1e-6)*scale, k^ = k/sqrt(|k|^2+1e-6),
 *   x = g_raw + g_bias[h], g = lower_bound*sigmoid(exp(A_log[h])*x) (bounded)
 *   or -exp(A_log[h])*softplus(x), beta = sigmoid(beta_raw),
 *   S <- S*diag(exp(g)); v' = beta*(v - S k^); S <- S + v' k^T; o = S q^.
 * Writes o (bf16, round to nearest even) to out[token][h][:], and the
 * token's record (raw: k, v, g_raw, beta_raw; correction: v', k, g_raw) to
 * record slot r = record_rows[b] (or b), position t.  The pool is NOT written, except by the deferred fold below.
 *
 * Deferred fold ([KIMI]: the next verify replays the pending count in the
 * same pass): if pending != NULL, r >= 0 and p = pending[r] > 0, the first p
 * records of slot r (the previous step's accepted tokens) are replayed from
 * the checkpoint first; the folded state is written back to state_pool[s][h]
 * and the new tokens run from it.  This happens even when T == 0.  pending is
 * read, never written: the commit after this step rewrites it.
 *
 * trajectory_out (tests only; NULL in production): fp32 [T_total][H][V][K],
 * the state after every token, i.e. what the full-state path would store.
 *
 * q, k, v, g_raw, beta_raw: bf16 inputs (see strides in cfg).
 * A_log: fp32 [H]; g_bias: fp32 [H * 128] (per channel).
 * out: bf16 [T_total][H][128], contiguous.  Rows that are skipped leave their
 * out entries and records untouched.
 * B: number of rows (B == 0: KDA_OK without a launch, and no pointer is
 * inspected, so empty tensors with NULL data pointers are accepted).
 */
kda_status kda_verify(const kda_config *cfg,
                      const void *q, const void *k, const void *v,
                      const void *g_raw, const void *beta_raw,
                      const float *A_log, const float *g_bias,
                      float *state_pool,
                      const int32_t *cu_seqlens, const int32_t *state_indices,
                      int32_t B,
                      const int32_t *record_rows, const int32_t *pending,
                      void *records, void *out, float *trajectory_out,
                      int32_t *error_word, void *stream);

/*
 * kda_commit -- fold each row's accepted tokens into its checkpoint
 * ([GLM] `_prepare_commit_plan_kernel` + `Glm5NextRecoverSSMCommitContext.commit`;
 * [KIMI] `KDADeferredCommitContext.commit` with record_rows/pending/eager).
 *
 * Per row: n = min(max(num_accepted[b], 0), T, Q); the row is valid iff
 * state_indices[b] > 0, n > 0 and its record slot r >= 0.
 * Eager mode (pending == NULL): a valid row replays its first n records from
 * state_pool[s][h] and writes the resulting state once (bit-identical to the
 * verify's trajectory state after its n-th token: same kernels, same order).
 * Deferred mode (pending != NULL): for every row with r >= 0, pending[r] is
 * set to n if the row is valid and not eager, else 0; rows with
 * eager[b] != 0 (eager may be NULL: no row) are committed now as above.
 * num_accepted: int32 [B].  eager: uint8 [B] or NULL.
 */
kda_status kda_commit(const kda_config *cfg,
                      const float *A_log, const float *g_bias,
                      float *state_pool,
                      const int32_t *cu_seqlens, const int32_t *state_indices,
                      int32_t B,
                      const int32_t *num_accepted,
                      const int32_t *record_rows, const void *records,
                      int32_t *pending, const uint8_t *eager,
                      int32_t *error_word, void *stream);

/*
 * kda_flush -- fold pending replays into the checkpoints in place
 * ([KIMI] `KDADeferredCommitContext.flush`), for a verify that does not fold
 * (pending == NULL) or before exporting a checkpoint.  For each row with
 * s > 0 and r >= 0 and p = pending[r] > 0, replays p records and writes the
 * state.  pending is left as it is; the commit after the next step rewrites it.
 * The rows' token counts play no part, so no cu_seqlens is taken.
 */
kda_status kda_flush(const kda_config *cfg,
                     const float *A_log, const float *g_bias,
                     float *state_pool,
                     const int32_t *state_indices, int32_t B,
                     const int32_t *record_rows, const void *records,
                     const int32_t *pending,
                     int32_t *error_word, void *stream);

/*
 * kda_conv_compact -- conv-state compaction of a commit ([GLM]
 * `_compact_conv_state_kernel` in its non-align form, launched by
 * `Glm5NextRecoverSSMCommitContext.commit` beside the state replay).
 *
 * The short causal conv in front of q, k and v keeps, per state slot, a
 * window of `width` columns per channel; after the verify it holds
 * [history[1:], x_0 .. x_{Q-1}] with history = width - Q + 1 columns.  For
 * each row b with T = cu_seqlens[b+1] - cu_seqlens[b], slot s =
 * state_indices[b] and n = min(max(num_accepted[b], 0), T, Q) (the commit's
 * count): if s > 0 and n > 0, every channel's columns [n-1, n-1+history) of
 * slot s move to columns [0, history), all read before any is written, so the
 * next step reads its history at column 0.  Columns from `history` on and all
 * other slots are left alone.  Deferred rows are compacted too: only the
 * recurrent replay is deferred, and the next step's conv needs the window now.
 * Rows with T outside [0, Q] or s >= num_slots are skipped and flagged in
 * *error_word (KDA_ROW_BAD_LENGTH, KDA_ROW_BAD_SLOT).
 *
 * conv_state: the caller's pool, element (slot, channel, column) at
 * slot*stride_slot + channel*stride_dim + column*stride_col elements of
 * elem_bytes each (2: bf16/fp16, 4: fp32; values are moved as bits).  Both
 * the channel-major ("dim first") and the column-major layouts are strides
 * of this form.  The strides must map distinct (channel, column) pairs of a
 * slot to distinct elements.  A separate launch from kda_commit: it runs
 * over every committed row, deferred or not, and is a plain copy.
 */
#define KDA_MAX_CONV_HISTORY 16

typedef struct kda_conv_config {
    int32_t num_slots;        /* S: slots of the conv-state pool (slot 0 = null) */
    int32_t conv_dim;         /* channels >= 1 */
    int32_t width;            /* columns per channel: history + window - 1 */
    int32_t window;           /* Q = 1 + num_spec, 1..8 */
    int32_t elem_bytes;       /* 2 or 4 */
    int32_t reserved;         /* 0 */
    int64_t stride_slot;      /* element strides, each >= 1 */
    int64_t stride_dim;
    int64_t stride_col;
} kda_conv_config;

kda_status kda_conv_compact(const kda_conv_config *cc, void *conv_state,
                            const int32_t *cu_seqlens, const int32_t *state_indices,
                            int32_t B, const int32_t *num_accepted,
                            int32_t *error_word, void *stream);

/*
 * Align mode ([GLM] `_prepare_commit_plan_kernel` with a block table,
 * `_replay_indices_kernel`, and the ALIGN_MODE branch of
 * `_compact_conv_state_kernel`): states live in paged blocks of block_size
 * tokens.  For a committing row with n accepted tokens, request q =
 * request_indices[b] (or b) and c = num_computed[q] tokens before this step:
 *   final block    = block_table[q][min((c + n - 1) / block_size, width - 1)];
 *   boundary       = (c / block_size + 1) * block_size, the first block
 *                    boundary after c; if c + n >= boundary the step reaches
 *                    it: boundary_len = boundary - c tokens and
 *                    boundary block = block_table[q][boundary / block_size - 1].
 * The state after n tokens (and the conv window at column n - 1) goes to the
 * final block; the state after boundary_len tokens (the conv window at column
 * boundary_len - 1) goes to the boundary block, for the recurrent state only
 * when boundary_len < n (otherwise the final block is that block).  Both are
 * computed from the row's source slot state_indices[b] as it was before the
 * call; the source is not written unless it is one of the blocks.  A row
 * whose final block is <= 0 commits nothing.  num_accepted is indexed by
 * request in align mode.  Rows must not write a block another row reads.
 */
typedef struct kda_align {
    const int32_t *block_table;      /* [num_requests][>= width], row stride below */
    int64_t block_table_stride;      /* elements between rows, >= width */
    int32_t block_table_width;       /* columns >= 1 */
    int32_t block_size;              /* tokens per block, >= window */
    int32_t num_requests;            /* rows of block_table, num_computed, num_accepted */
    int32_t reserved;                /* 0 */
    const int32_t *num_computed;     /* [num_requests] */
    const int32_t *request_indices;  /* [B], or NULL: request b is row b */
} kda_align;

/*
 * kda_commit_align -- the commit in align mode: as kda_commit, but the
 * replayed states go to the final and boundary blocks above.  Rows with a
 * request index outside [0, num_requests), a negative num_computed or a
 * boundary block past the table are skipped and flagged KDA_ROW_BAD_BLOCK; a
 * block >= num_slots flags KDA_ROW_BAD_SLOT.  num_accepted: int32
 * [num_requests].
 *
 * pending == NULL: every valid row is committed now (eager).
 * pending != NULL (the deferred commit of [KIMI] `KDADeferredCommitContext.commit`
 * with a block table): a valid row is committed now when eager[b] != 0
 * (eager may be NULL: no row), when its final block is not its own state
 * slot state_indices[b], or when it owes a boundary block (boundary_len <
 * n); its pending[r] is set to 0.  Any other valid row only sets pending[r]
 * = n: its final block is its own slot and no boundary state is due, so the
 * next verify's fold (or kda_flush), which stores to the row's slot, leaves
 * exactly what this commit would have written.  Rows that commit nothing,
 * and rows skipped for bad metadata whose record slot is in range, get
 * pending[r] = 0.  The pages leave the fold's target in align mode open;
 * this rule is the reading that keeps every block right.
 */
kda_status kda_commit_align(const kda_config *cfg,
                            const float *A_log, const float *g_bias,
                            float *state_pool,
                            const int32_t *cu_seqlens, const int32_t *state_indices,
                            int32_t B,
                            const int32_t *num_accepted,
                            const int32_t *record_rows, const void *records,
                            const kda_align *align,
                            int32_t *pending, const uint8_t *eager,
                            int32_t *error_word, void *stream);

/*
 * kda_conv_compact_align -- kda_conv_compact in align mode: the window at
 * column n - 1 of the source slot goes to columns [0, history) of the final
 * block, and the window at column boundary_len - 1 to the boundary block when
 * the step reaches one; both windows are read before either is written.
 * num_accepted: int32 [num_requests].
 */
kda_status kda_conv_compact_align(const kda_conv_config *cc, void *conv_state,
                                  const int32_t *cu_seqlens, const int32_t *state_indices,
                                  int32_t B, const int32_t *num_accepted,
                                  const kda_align *align,
                                  int32_t *error_word, void *stream);

/*
 * kda_record_state_blocks -- the align-mode bookkeeping after a commit
 * (recoverssm.py, `_record_state_block_kernel` and `record_state_blocks`,
 * run from the runner's commit hook): each committed request's running
 * state column is pointed at the block that holds its last committed token,
 * where kda_commit_align left its state, and its accepted count is reset to
 * 1, so that the next step's pre-step copy reads the state from there.  For
 * each spec row i in [0, B):
 *   q    = align->request_indices[i] (NULL: q = i)
 *   s    = idx_mapping[q], the request's index in the running arrays;
 *          s < 0: nothing is recorded for the row
 *   last = max(align->num_computed[q] + num_sampled[q] - 1, 0)
 *   state_column[s] = min(last / align->block_size, align->block_table_width - 1)
 *   num_accepted[s] = 1
 * With num_sampled[q] equal to the commit count n of the row, state_column[s]
 * is the column of the final block in kda_commit_align.
 *
 * align: block_size >= 1, block_table_width >= 1, num_requests >= 1 and
 *   num_computed are read; block_table and block_table_stride are not (the
 *   descriptor passed to kda_commit_align can be reused as it is).
 * idx_mapping, num_sampled: int32 [num_requests], device.
 * state_column, num_accepted: int32 [num_states], device, written for the
 *   rows' s only; num_states >= 1.
 * Device-detected bad data: q outside [0, num_requests) flags
 * KDA_ROW_BAD_BLOCK, s >= num_states flags KDA_ROW_BAD_SLOT; the row is
 * skipped.  Two rows with the same s are the caller's error (one of the two
 * writes wins).  B == 0: KDA_OK, nothing inspected or launched.  A host check
 * above that fails (or a NULL or misaligned pointer) returns
 * KDA_ERR_INVALID_ARG.  One thread per row, one launch on `stream`.
 */
kda_status kda_record_state_blocks(const kda_align *align,
                                   const int32_t *idx_mapping, const int32_t *num_sampled,
                                   int32_t B,
                                   int32_t *state_column, int32_t *num_accepted,
                                   int32_t num_states,
                                   int32_t *error_word, void *stream);

/* Name of a status code (static string). */
const char *kda_status_string(kda_status status);

/* ABI version of this header: bumped on any signature or layout change. */
int32_t kda_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_KDA_H */

/*
 * lora.h — C ABI of the GB300 (sm_103a) LoRA linear layer.
 *
 * The layer, as the LoRAFusion write-ups state it (Eurosys26 LoRAFusion
 * article, juhe.plus, section 2 "background"; LoRAFusion notes,
 * papers.chlience.com, section 5 "FusedLoRA" / "FusedMultiLoRA"):
 *
 *     Y = X W + alpha * (dropout(X) A) B = X W + alpha * S B,   S = X_hat A
 *
 * with W frozen and only A, B trained.  Shapes: X m x k, W k x n, A k x r,
 * B r x n, Y m x n.  Every matrix is row-major bf16 (its bit pattern passed
 * as uint16_t) unless stated otherwise.  Arithmetic accumulates in fp32.
 *
 * Dropout (the pages fix no generator; the reading taken here): inverted
 * dropout on the branch input, kept elements scaled by q = 1/(1-p).  The keep
 * decision of element (t, j) — t the global row of the packed batch, j the
 * feature — is lane j%8 of Philox4x32-10 (Salmon et al., SC'11) with key
 * (seed low word, seed high word) and counter (t, j/8, 0, 0): the four
 * output words give eight 16-bit lanes, low half first, and the element is
 * kept iff lane >= T, T = floor(p*65536 + 0.5).  The backward regenerates
 * the decisions from the seed, so the calls need share nothing but S_saved;
 * a caller may instead keep the bits the forward writes (mask_bits) and hand
 * them to the backward, which then reads them (same decisions, less work).
 *
 * Multi-adapter form (LoRAFusion notes, section 5 "FusedMultiLoRA"; article
 * section 4.1): rows are grouped in 128-row tiles; a segment table assigns
 * each tile to one adapter (A_i, B_i, alpha_i, p_i); the frozen product X W
 * is shared by every row, the branch of a tile uses its own adapter, and the
 * gradients of each adapter sum over that adapter's rows only.  Rows that no
 * segment covers get no branch (Y = X W, dX = dY W^T there).
 *
 * Conventions for every entry point below:
 *  - Device pointers are device memory of the current CUDA device; the caller
 *    owns every buffer.  The library never allocates or frees memory.
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the call returns without synchronising.  A kernel that gives
 *    up on a bounded internal wait records a code in the workspace; read it
 *    with lora_device_status().
 *  - Validation happens before any launch; a failing call enqueues nothing
 *    and returns a status.  Nothing is thrown across this interface.
 *  - k and n must be multiples of 8 in [8, 2^24], ranks multiples of 8 in
 *    [8, 128], every pointer 16-byte aligned, 0 <= p < 1, m <= 262144 rows.
 *  - Gradients dA, dB are overwritten, not accumulated.
 *  - `workspace` is device memory of at least lora_workspace_size() bytes,
 *    256-byte aligned, filled with zeros before its first use (cudaMemset).
 *    Every call that completes leaves it zeroed again; after a call reports
 *    LORA_EDEVICE_TIMEOUT, zero it before reusing it.  One workspace must not
 *    be used by two calls that may run concurrently.
 *  - Host threads may call any entry point at the same time: every call
 *    prepares its launches in storage of its own thread, and no call holds a
 *    lock while it enqueues work.  Calls on different streams with different
 *    workspaces are independent on the GPU too: the backward's side stream
 *    (below) belongs to the caller's stream.
 *  - When the backward regenerates the keep mask (no mask_bits given) and
 *    k % 128 == 0, the dX GEMM writes the decisions it regenerates for its
 *    own epilogue into the workspace and the dA pass reads them after it.
 *    Otherwise the backward forks its dA pass onto a side stream, beside the
 *    dX GEMM, and joins it back to `stream` before it returns work to it; the
 *    first such call on a stream creates that stream's side stream and two
 *    events: make it before any stream capture.
 */
#ifndef LORA_GB300_H
#define LORA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t lora_bf16; /* bfloat16 bit pattern */

typedef enum {
    LORA_OK = 0,
    LORA_EINVAL = 1,          /* missing pointer, p outside [0,1), rank outside [8,128], ... */
    LORA_EALIGN = 2,          /* a pointer is not 16-byte aligned (workspace: 256) */
    LORA_ESHAPE = 3,          /* k or n not a multiple of 8 or above 2^24, m too large, empty k or n */
    LORA_EARCH = 4,           /* the current device is not an sm_103 GPU */
    LORA_ECUDA = 5,           /* a CUDA runtime or driver call failed */
    LORA_EWORKSPACE = 6,      /* workspace missing, misaligned or too small */
    LORA_EDEVICE_TIMEOUT = 7, /* a kernel gave up on a bounded wait (from lora_device_status) */
    LORA_ETABLE = 8           /* segment table invalid: overlap, misalignment, bad adapter id */
} lora_status;

enum { LORA_TILE_ROWS = 128, LORA_MAX_RANK = 128, LORA_MAX_ADAPTERS = 16, LORA_MAX_ROWS = 262144,
       LORA_MAX_FEATURES = 16777216 /* k and n */ };

/* One adapter of the multi-adapter form.  A_i is k x rank, B_i is rank x n;
 * dA_i / dB_i (same shapes) are written by multi_lora_bwd and may be NULL
 * for multi_lora_fwd. */
typedef struct {
    int32_t rank;
    float alpha;
    float p;
    const lora_bf16* A;
    const lora_bf16* B;
    lora_bf16* dA;
    lora_bf16* dB;
} lora_adapter;

/* Rows [row_start, row_start + rows) use adapter `adapter`.  row_start is a
 * multiple of 128; rows is a multiple of 128 unless the segment ends at row m.
 * Segments must not overlap.  (Padding rows inside a segment are ordinary
 * rows: callers that pad samples to whole tiles put zeros there.) */
typedef struct {
    int64_t row_start;
    int64_t rows;
    int32_t adapter;
    int32_t reserved;
} lora_segment;

/* Workspace bytes sufficient for every call below with these sizes
 * (r_max: the largest rank; n_adapters: adapters per call, >= 1), in the
 * current reduction mode (lora_set_deterministic): the deterministic mode
 * needs a larger workspace, sized for the current device.
 *
 * The last region of this size holds the partial sums of GEMM output tiles
 * whose K loop is split over several CTA pairs (up to 80 pairs x 256 KB, 21
 * MB; less when the GEMMs have few tiles).  A call whose workspace ends before
 * that region still runs, with every tile computed whole by one pair: the GEMMs
 * then leave more CTA pairs idle when their last wave of tiles is nearly empty.
 * Results with and without the region agree to fp32 rounding; the split sums
 * are added in a fixed order, so either form is bit-reproducible in the
 * deterministic mode. */
size_t lora_workspace_size(int64_t m, int64_t k, int64_t n, int32_t r_max, int32_t n_adapters);

/* Reduction mode of every later call in this process (0 by default).
 *
 * The rank-r passes split their sums over many CTAs: S over the features
 * of each token tile, dS over n, dA over the tokens of each adapter, dB over
 * the tokens.  In the default mode (0) each CTA adds its partial into an fp32
 * accumulator with hardware reductions, whose order varies from call to
 * call, so the low bits of S_saved, dX, dA and dB may differ between two
 * calls on the same inputs (the keep mask and the routing never do).
 *
 * Mode 1 makes every output of lora_fwd, lora_bwd, multi_lora_fwd and
 * multi_lora_bwd bit-identical from call to call on the same device and
 * sizes (the LoRAFusion notes, papers.chlience.com, list the seed and the
 * mixed precision among the things a run should be able to re-check): each
 * CTA writes its partial of S, dS and dA to a slot of its own in the
 * workspace and the finalize passes add an item's slots in CTA order; dB is
 * computed in a second read of dY in which every dB element is the sum of at
 * most two partials onto zero (fp32 addition of two terms commutes exactly).
 * Cost: the second read of dY and a larger workspace.  Set the mode before
 * sizing workspaces and between calls; a call sizes its work by the mode it
 * finds.  DoRA's norm and dmag reductions stay atomic in both modes.
 * LORA_EINVAL unless `on` is 0 or 1. */
lora_status lora_set_deterministic(int32_t on);
int32_t lora_get_deterministic(void);

/* Forward, one adapter.  Writes Y (m x n), S_saved (m x r: alpha * S in bf16,
 * opaque state for lora_bwd) and, if mask_bits is not NULL (16-byte
 * aligned, m x k/8 bytes), the keep decisions: bit j%8 of byte t*(k/8) + j/8.
 * Steps (article section 4.1, forward ① and ②): dropout fused with the
 * down-projection, then X W + alpha S B as one contraction [X | alpha S][W; B]. */
lora_status lora_fwd(const lora_bf16* X, const lora_bf16* W, const lora_bf16* A, const lora_bf16* B,
                     float alpha, float p, uint64_t seed, int64_t m, int64_t k, int64_t n, int32_t r,
                     lora_bf16* Y, lora_bf16* S_saved, uint8_t* mask_bits,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Backward, one adapter, W frozen.  Inputs: dY (m x n), the forward's X, W,
 * A, B, S_saved and the same alpha, p, seed.  Writes
 *   dX = dY W^T + (D q) * (dS A^T),  dA = X_hat^T dS,  dB = alpha S^T dY,
 * with dS = alpha dY B^T (article section 4.1, backward ③ and ⑤).
 * mask_bits (optional, 16-byte aligned): the keep bits the forward wrote with
 * the same X, seed and p.  When given, the backward reads the mask instead of
 * regenerating it (the results are the same; the dX GEMM uses them when
 * k % 32 == 0, the dA pass when k % 128 == 0).  NULL: the mask is
 * regenerated from the seed. */
lora_status lora_bwd(const lora_bf16* dY, const lora_bf16* X, const lora_bf16* W, const lora_bf16* A,
                     const lora_bf16* B, const lora_bf16* S_saved, const uint8_t* mask_bits, float alpha, float p,
                     uint64_t seed, int64_t m, int64_t k, int64_t n, int32_t r, lora_bf16* dX, lora_bf16* dA,
                     lora_bf16* dB, void* workspace, size_t workspace_bytes, void* stream);

/* Forward, packed multi-adapter batch.  `adapters` and `segments` are HOST
 * arrays, read before the call returns.  S_saved is m x s_ld with
 * s_ld = the largest adapter rank; row t of adapter i holds alpha_i S in
 * columns [0, r_i) and zeros after; rows without an adapter are not written.
 * mask_bits (optional) is written for rows that have an adapter.
 * n_adapters may be 0 only with n_segments == 0 (the frozen layer alone). */
lora_status multi_lora_fwd(const lora_bf16* X, const lora_bf16* W, const lora_adapter* adapters, int32_t n_adapters,
                           const lora_segment* segments, int32_t n_segments, uint64_t seed, int64_t m, int64_t k,
                           int64_t n, lora_bf16* Y, lora_bf16* S_saved, uint8_t* mask_bits,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Backward of multi_lora_fwd.  Writes dX (m x k) and every adapter's dA_i,
 * dB_i (adapters without rows get zeros).  mask_bits: optional, as lora_bwd
 * (the bits multi_lora_fwd wrote for the same batch). */
lora_status multi_lora_bwd(const lora_bf16* dY, const lora_bf16* X, const lora_bf16* W, const lora_adapter* adapters,
                           int32_t n_adapters, const lora_segment* segments, int32_t n_segments, uint64_t seed,
                           int64_t m, int64_t k, int64_t n, const lora_bf16* S_saved, const uint8_t* mask_bits,
                           lora_bf16* dX, void* workspace, size_t workspace_bytes, void* stream);

/* DoRA ("Scaling DoRA", paper.rainbus.top): the adapted weight split into a
 * magnitude per output feature and a direction,
 *     W' = mag * (W + alpha A B) / ||W + alpha A B||  (norm over each column j),
 *     Y  = g * (X W + alpha (dropout(X) A) B),  g_j = mag_j / ||W_j + alpha (A B)_j||,
 * in this layer's orientation (W k x n, so the n output features are columns).
 * The norm comes from the pages' factored identity
 *     ||W_j||^2 + 2 alpha B_j . (W^T A)_j + alpha^2 B_j^T (A^T A) B_j,
 * never from the dense k x n update.  Single adapter; rank, p, alignment and
 * shape rules as for lora_fwd.  mag, w_norm2, g_saved and dmag are fp32
 * vectors of n, 16-byte aligned.  Every mag_j must be finite and nonzero:
 * dora_bwd recovers dmag from Y by dividing by mag_j (Y's column j is zero
 * when mag_j is, and the gradient could not be recovered from it); the
 * library does not read mag on the host, so it cannot check this. */

/* Workspace bytes for dora_fwd / dora_bwd: lora_workspace_size(m, k, n, r, 1)
 * plus the DoRA accumulators (W^T A, A^T A, dmag).  Same contract as the LoRA
 * workspace: zero before the first call, and every completed call leaves it
 * zero. */
size_t dora_workspace_size(int64_t m, int64_t k, int64_t n, int32_t r);

/* w_norm2[j] = ||W[:, j]||^2 in fp32 (W k x n is frozen: compute once and
 * pass to every dora_fwd).  Asynchronous on `stream`. */
lora_status dora_weight_norm2(const lora_bf16* W, int64_t k, int64_t n, float* w_norm2, void* stream);

/* DoRA forward: writes Y (m x n), S_saved (as lora_fwd), g_saved (n: the
 * column scale, needed by dora_bwd) and optionally mask_bits. */
lora_status dora_fwd(const lora_bf16* X, const lora_bf16* W, const lora_bf16* A, const lora_bf16* B, const float* mag,
                     const float* w_norm2, float alpha, float p, uint64_t seed, int64_t m, int64_t k, int64_t n,
                     int32_t r, lora_bf16* Y, lora_bf16* S_saved, float* g_saved, uint8_t* mask_bits, void* workspace,
                     size_t workspace_bytes, void* stream);

/* DoRA backward with the column norm held constant (as DoRA trains; the pages
 * fix no backward): dZ = dY * g feeds the LoRA backward, giving dX, dA, dB;
 * dmag_j = sum_t dY[t, j] Y[t, j] / mag_j (= sum_t dY Z / ||.||_j).  Inputs
 * are the forward's X, W, A, B, S_saved, Y, mag, g_saved and the same alpha,
 * p, seed.  mask_bits: optional, as lora_bwd (the bits dora_fwd wrote).
 * dZ: caller scratch of m x n bf16 (16-byte aligned; its contents before and
 * after the call do not matter). */
lora_status dora_bwd(const lora_bf16* dY, const lora_bf16* X, const lora_bf16* W, const lora_bf16* A,
                     const lora_bf16* B, const lora_bf16* S_saved, const uint8_t* mask_bits, const lora_bf16* Y,
                     const float* mag,
                     const float* g_saved, float alpha, float p, uint64_t seed, int64_t m, int64_t k, int64_t n,
                     int32_t r, lora_bf16* dX, lora_bf16* dA, lora_bf16* dB, float* dmag, lora_bf16* dZ,
                     void* workspace, size_t workspace_bytes, void* stream);

/* lora_fwd for callers that cannot allocate device memory (no counterpart in
 * the LoRAFusion write-ups; it only changes where the scratch lives).
 * Some callers have no way to hand the library a workspace: a plugin whose
 * host application plans every device buffer ahead of time and offers none
 * to extensions, or a runtime that forbids allocation on its compute path.
 * This entry point takes the same arguments as lora_fwd minus the workspace
 * and uses a file-scope device array of LORA_STATIC_SCRATCH_BYTES (8 MiB)
 * inside the library instead; every GPU that loads the library keeps that
 * array until the process exits.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *  - Sizes whose scratch need (lora_workspace_size(m, k, n, r, 1)) exceeds
 *    8 MiB are rejected with LORA_EWORKSPACE and lora_last_error_string()
 *    says why.  For example m = 8192, k = 4096, n = 14336, r = 16 needs 2 MB.
 *  - Arguments are checked exactly as lora_fwd checks them, and before
 *    anything is enqueued: a call that returns an error has enqueued nothing.
 *  - The first successful call on each device looks up the array's device
 *    address and clears the whole array, on `stream`; make that first call
 *    before any stream capture.
 *  - Every call on a device shares the one array and leaves its contents
 *    behind.  Every call that completes leaves its accumulators and counters
 *    at zero again, so the next call (of any shape) starts clean.  Calls whose work can overlap on the GPU
 *    (different streams, no ordering) race on the array.
 *  - Bounded-wait timeouts are recorded in the array's status word, which no
 *    entry point reads back; a call that timed out may leave the array dirty,
 *    and later results on that device are then not to be trusted. */
enum { LORA_STATIC_SCRATCH_BYTES = 8 << 20 };
lora_status lora_fwd_static_scratch(const lora_bf16* X, const lora_bf16* W, const lora_bf16* A, const lora_bf16* B,
                                    float alpha, float p, uint64_t seed, int64_t m, int64_t k, int64_t n, int32_t r,
                                    lora_bf16* Y, lora_bf16* S_saved, uint8_t* mask_bits, void* stream);

/* Host only, no GPU needed: the routing table.  tile_adapter[i] (i < ceil(m/128))
 * receives the adapter of tile i, -1 where no segment covers it. */
lora_status lora_tile_table(const lora_segment* segments, int32_t n_segments, int32_t n_adapters, int64_t m,
                            int32_t* tile_adapter, int64_t n_tiles);

/* Host only: the keep threshold T for drop rate p (LORA_EINVAL outside [0,1)). */
lora_status lora_keep_threshold(float p, uint32_t* T);

/* Host only, no GPU needed: greedy token-capacity packing of samples into
 * microbatches, the fallback packer of the LoRAFusion multi-adapter scheduler
 * (notes on papers.chlience.com, section 5 "Multi-LoRA scheduler"; article,
 * section 4.2 step 2).  First-fit decreasing: a sample occupies its length
 * rounded up to whole 128-row tiles; samples are taken longest first (equal
 * sizes in sample order) and each goes into the first microbatch, in opening
 * order, with room left, else into a new one.
 *   lengths[i]          tokens of sample i (>= 1), host array of n_samples
 *   capacity            rows per microbatch, a positive multiple of 128
 *   batch_of_sample[i]  receives the microbatch of sample i (0-based)
 *   row_of_sample[i]    receives its first row there (samples of a microbatch
 *                       lie back to back from row 0 in placement order)
 *   *n_batches          receives the number of microbatches
 * The samples of microbatch b with their rows and adapters form the segment
 * table of a multi_lora_fwd / multi_lora_bwd call.  LORA_EINVAL for missing
 * pointers, a length below 1 or a bad capacity; LORA_ESHAPE if a sample does
 * not fit in one microbatch.  Nothing is written when the call fails. */
lora_status lora_pack_greedy(const int64_t* lengths, int32_t n_samples, int64_t capacity,
                             int32_t* batch_of_sample, int64_t* row_of_sample, int32_t* n_batches);

/* Synchronises `stream`, then reads and clears the device status word of
 * `workspace`.  *code receives the raw device code (0 = none).  Returns
 * LORA_EDEVICE_TIMEOUT if a kernel gave up on a bounded wait. */
lora_status lora_device_status(void* workspace, void* stream, int32_t* code);

/* Sets the bound, in nanoseconds, after which a kernel stops waiting on an
 * internal barrier, records LORA_EDEVICE_TIMEOUT and returns (default 2 s). */
void lora_set_wait_limit_ns(uint64_t ns);

/* Test hook for the bounded waits: launches one kernel that waits on a
 * barrier nothing will complete, with the current limit, and returns.  The
 * device status then reads LORA_EDEVICE_TIMEOUT; the context stays usable. */
lora_status lora_debug_stuck_wait(void* workspace, size_t workspace_bytes, void* stream);

/* Test hook for the schedule of the CTA-pair GEMMs (host only; no device is
 * needed).  For an M x N output in tiles of 256 rows x bn columns, `stages`
 * 64-deep K stages a tile, at most `max_pairs` CTA pairs (half the SMs),
 * tile splitting allowed (allow_split != 0) or not, and one accumulator set
 * per CTA (single_acc != 0: the 256-wide backward GEMM) or two, *pairs
 * receives the grid's pair count and *split_tiles the number of tiles split
 * by K.  Run i of the schedule is written to runs[4i .. 4i+3] as (pair, tile,
 * first stage, end stage) for i < cap, pairs in order and each pair's runs in
 * the order it works through them; *n_runs receives the number of runs.  A
 * split tile's stages are spread over several runs: the run holding stage 0
 * adds the others' partial sums and stores the tile.  LORA_EINVAL for
 * missing pointers or arguments below 1 (cap below 0). */
lora_status lora_debug_gemm_runs(int64_t M, int64_t N, int32_t bn, int32_t stages, int32_t max_pairs,
                                 int32_t allow_split, int32_t single_acc, int32_t* pairs, int32_t* split_tiles,
                                 int32_t* runs, int64_t cap, int64_t* n_runs);

const char* lora_status_string(lora_status s);

/* Measurement: between lora_timing_begin() and lora_timing_end(), every
 * kernel (and workspace memset) the library enqueues is bracketed by CUDA
 * events on its own stream.  lora_timing_end() waits for those events and
 * fills, for each kind i < n_kinds (see lora_kernel_name), the summed device
 * time in ms and the number of launches.  Kinds: 0 down-projection,
 * 1 finalize S, 2 forward GEMM, 3 dS/dB, 4 finalize dS/dB, 5 backward GEMM,
 * 6 dA, 7 finalize dA, 8 memset (gradients of adapters that own no rows),
 * 9-12 DoRA (U, norm, dZ, dmag).  When kind 6 runs on the library's side
 * stream beside the backward GEMM, its event pair spans from the fork to its
 * end.
 * Host-side cost: two event records per launch. */
enum { LORA_KERNEL_KINDS = 13 };
lora_status lora_timing_begin(void);
lora_status lora_timing_end(float* total_ms, int32_t* launches, int32_t n_kinds);
const char* lora_kernel_name(int32_t kind);

/* Host only: the CUDA error text behind the calling thread's last LORA_ECUDA
 * (a static string; "no error" if none occurred). */
const char* lora_last_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* LORA_GB300_H */

/*
 * w4a16.h — C ABI of the GB300 (sm_103a) W4A16 group-32 decode library.
 *
 * Format (page "Gemma 4 on a 4 GB GPU in Plain PyTorch", sections "Step 1 —
 * Load Google's QAT Weights Without Unpacking Them" and "Step 3 — Multiply
 * Straight From the Packed Weights"): a weight matrix W of N rows by K columns
 * is stored as 4-bit codes in groups of 32 along K, with one 16-bit step per
 * group, and W[n][k] = (code[n][k] - 8) * step[n][k / 32].  Activations and
 * outputs are 16-bit.  Concretely, in this library:
 *
 *   qw  uint32 [N][K/8]  row-major; element k of row n is the 4-bit field at
 *                        bits 4*(k%8) .. 4*(k%8)+3 of word k/8 (low nibble
 *                        first);
 *   st  bf16   [N][K/32] row-major steps;
 *   x   bf16   [M][K]    row-major activations;
 *   y   bf16   [M][N]    row-major results, y[m][n] = sum_k W[n][k] * x[m][k]
 *                        accumulated in fp32 and rounded to nearest-even once.
 *
 * Conventions shared by every call:
 *   - All array pointers are DEVICE pointers owned by the caller.  Calls only
 *     enqueue work on `stream` (a cudaStream_t; 0 = legacy default stream) and
 *     return; they never synchronise and never allocate device memory.
 *   - Argument errors that the host can see (null pointers, sizes, alignment)
 *     return a w4_status != W4_OK BEFORE any launch, and no output is touched.
 *   - Errors that only the device can see (an id out of range, a wait that
 *     timed out) are written into *status_dev, a caller-owned device int32
 *     that the caller zeroes beforehand and reads after synchronising; the
 *     first error recorded stays.  The output rows concerned are left
 *     UNWRITTEN, so a caller that pre-fills its output can tell a failed row
 *     from a result (page "Fixing Gemma 4's oversized KV cache", section "A
 *     failed decode must not look uncertain": an untouched zero row passed
 *     for a valid answer).  status_dev may be NULL; then such errors are
 *     visible only through the unwritten rows.
 *   - W4_FLAG_PDL launches the kernel as a programmatic dependent of the
 *     previous kernel in the stream: its weight loads may start before that
 *     kernel has finished, and it waits for it before reading activations or
 *     ids and before writing any output.  Use it only when nothing still
 *     running earlier in the stream writes qw / st.
 *   - Results are deterministic: the same inputs give the same bits on every
 *     call, and the arithmetic of an output row depends only on K, on the
 *     path that computes it, on that row's codes and steps and on its
 *     activation row (not on N, the row index, the number of ids or the
 *     addresses), so w4a16_gemv_id row i is bitwise equal to w4a16_gemv on
 *     expert ids[i] with the same activation row.
 *   - Two paths compute w4a16_gemv.  The CUDA-core path (every w4a16_gemv_id
 *     call, and w4a16_gemv with 1 or 2 activation rows, or 3 to 4 rows of
 *     small weights) dequantises in packed fp16 with fp16 partial sums of 4
 *     products; its rows do not depend on M.  The tensor-core path
 *     (w4a16_gemv with 5 or more rows, 4 rows when N * K >= 2^24, 3 rows
 *     when N * K >= 2^27, K a multiple of 256) lets tcgen05 MMAs take exact bf16 products with
 *     fp32 sums: up to 32 rows it folds each group's step into the sum after
 *     the MMA, from 33 rows (prompt chunks) it splits each weight exactly
 *     into two bf16 parts and accumulates over the whole of K.  Within
 *     each of these kernels rows do not depend on M; the kernels differ from
 *     each other in the last bits.  W4_FLAG_CUDA_CORES or
 *     W4_FLAG_TENSOR_CORES pins the path.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Identical to cudaStream_t. */
typedef struct CUstream_st *w4_stream_t;

typedef enum w4_status {
    W4_OK = 0,
    W4_ERR_ARG = 1,        /* null pointer, size < 1, unknown flag bit */
    W4_ERR_ALIGN = 2,      /* pointer or stride breaks its alignment rule */
    W4_ERR_SHAPE = 3,      /* K not a multiple of 32 or above the maximum, M or
                              x_rows outside the supported range */
    W4_ERR_WORKSPACE = 4,  /* workspace smaller than w4a16_gemv_workspace_bytes */
    W4_ERR_LAUNCH = 5,     /* the CUDA launch failed */
    W4_ERR_INDEX = 6,      /* device-side: an id outside [0, count) */
    W4_ERR_VALUE = 7,      /* device-side: a code outside 0..15 (w4_pack) */
    W4_ERR_TIMEOUT = 8,    /* device-side: a bounded wait in a kernel expired */
    W4_ERR_DEVICE = 9,     /* no usable CUDA device / attribute query failed */
    W4_ERR_STATE = 10,     /* slot pool: request cannot be served, or a pool
                              copy failed (the pool forgot the experts it was
                              loading) */
    W4_ERR_OWNER = 11      /* device-side: a slot does not hold the expert
                              named for it (w4a16_gemv_id_scaled) */
} w4_status;

#define W4_FLAG_PDL 1u
#define W4_FLAG_CUDA_CORES 2u     /* w4a16_gemv: CUDA-core path at any M */
#define W4_FLAG_TENSOR_CORES 4u   /* w4a16_gemv: tensor-core path at any M (K % 256 == 0) */
#define W4_FLAG_SILU_MUL 8u       /* w4a16_gemv: x rows are [gate K | up K]; the product
                                     takes h = silu(gate) * up (CUDA-core path) */
#define W4_FLAG_IDS_FINAL 16u     /* w4a16_gemv_id(_scaled) with W4_FLAG_PDL: ids were
                                     written before the previous kernel in the stream
                                     began (e.g. the slot ids of the layer's previous
                                     routed call); the copy warps then read them and start
                                     the weight copies before the dependency wait
                                     (activations, real ids and the slot table are still
                                     read after it) */

#define W4_GROUP 32        /* codes per group along K */
#define W4_MAX_K 65536     /* largest supported K */
/* Largest batch of activation rows per call: a prompt chunk of 256 tokens
 * (page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 6 — Read
 * Prompts in 32-Bit on a Card Without Tensor Cores"). */
#define W4_MAX_M 256
#define W4_ABI_VERSION 4

/* Human-readable name of a status code (static string). */
const char *w4_status_str(int status);

/* W4_ABI_VERSION of the loaded library. */
int w4_abi_version(void);

/* Text of the CUDA error behind the calling thread's last W4_ERR_LAUNCH or
 * W4_ERR_STATE from a failed enqueue ("no error" if none; static string). */
const char *w4_last_cuda_error(void);

/*
 * w4a16_gemv — dense W4A16 matrix-vector (or small-batch matrix) product.
 *
 * Page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 3 — Multiply
 * Straight From the Packed Weights": each decoded token needs the product of
 * an activation vector with each weight matrix, taken from the packed 4-bit
 * words as they are stored.
 *
 *   y[m][n] = bf16( sum_{k<K} (code[n][k] - 8) * st[n][k/32] * x[m][k] )
 *
 * y          bf16 [M][N], written once per element (2-byte aligned).
 * qw         uint32 [N][K/8], 16-byte aligned.
 * st         bf16 [N][K/32], 16-byte aligned.
 * x          bf16 [M][K], 16-byte aligned.
 * M          1 .. W4_MAX_M activation rows.  By default (K a multiple of
 *            256): 1-2 rows, and 3-4 rows of small weights (N * K below 2^27
 *            at 3 rows, below 2^24 at 4), the CUDA-core path; other batches up
 *            to 32 rows one launch of the tensor-core small-batch kernel (the
 *            CUDA-core path for every M up to 32 when K is not a multiple of
 *            256, one launch per 4 rows); 33 to W4_MAX_M rows (a
 *            prompt chunk) one launch of the tensor-core GEMM.  A call pinned
 *            to the CUDA cores enqueues one launch per 4 rows at any M (each
 *            reading the weights), all checked before the first is
 *            enqueued.
 * N          >= 1 output rows.
 * K          multiple of 32, 32 .. W4_MAX_K.
 * workspace  device scratch of at least w4a16_gemv_workspace_bytes(M, N, K)
 *            bytes (16-byte aligned), or NULL when that is 0.  It must be
 *            zero-filled before its first use; every call that completes
 *            without a device-side error leaves it zero-filled again.  Calls
 *            that may run concurrently need separate workspaces.  On the
 *            tensor-core small-batch path a call whose row tiles do not
 *            divide evenly over the CTAs uses the workspace for balanced runs
 *            (w4_plan_info.dynamic_windows); given less (or NULL) it runs the
 *            plain plan instead, with the same bits, and returns an error only
 *            when a K split needs the workspace.
 * status_dev device int32 for device-side errors (W4_ERR_TIMEOUT), or NULL.
 * flags      W4_FLAG_PDL, and at most one of W4_FLAG_CUDA_CORES /
 *            W4_FLAG_TENSOR_CORES (default: the rule under M above;
 *            W4_ERR_SHAPE if the pinned path cannot run K).
 *            W4_FLAG_SILU_MUL: the gated MLP's down projection fused with its
 *            activation (page "Gemma 4 on a 4 GB GPU in Plain PyTorch", tip
 *            "Merge the Small Projections": gate and up are one merged GEMV,
 *            whose output row [gate | up] feeds this call directly).  x is
 *            then [M][2K] bf16 and the GEMV multiplies
 *            h[m][k] = gate[m][k] / (1 + e^-gate[m][k]) * up[m][k], computed
 *            in fp32 while the activations are staged (no bf16 rounding of h,
 *            no separate kernel); CUDA-core path at any M (with
 *            W4_FLAG_TENSOR_CORES: W4_ERR_SHAPE).
 * Returns W4_OK once the work is enqueued.
 *
 * Large CUDA-core launches (w4_plan_info.dynamic_windows) hand their row
 * windows to the CTAs from a counter held by the library: one of 1024 slots
 * per device, taken round robin per launch and re-armed by the launch's last
 * CTA.  Only a launch still running 1024 launches after it was enqueued (on
 * any stream of the device) could meet its slot in use.
 */
w4_status w4a16_gemv(void *y, const void *qw, const void *st, const void *x,
                     int M, int N, int K, void *workspace, size_t workspace_bytes,
                     int32_t *status_dev, unsigned flags, w4_stream_t stream);

/* Scratch bytes to give w4a16_gemv for this shape with flags 0: enough for
 * every launch a call of this shape makes (on the CUDA cores, the largest
 * split-K scratch of the plans for up to 4 rows, so it may exceed what one
 * launch uses); 0 when none of them splits K. */
size_t w4a16_gemv_workspace_bytes(int M, int N, int K);

/* The same for a call with the given flags (path flags change the plan). */
size_t w4a16_gemv_workspace_bytes_flags(int M, int N, int K, unsigned flags);

/*
 * w4a16_gemv_prefetch_l2 — w4a16_gemv that also brings the next call's
 * weights into L2 while it finishes.
 *
 * Page "Running a 26B MoE on an 8 GB Jetson by streaming experts from SSD",
 * section on hiding the expert reads: the reads for the next piece of work
 * are started while the GPU computes work it had to do anyway, and are
 * joined only where that data is needed.  On GB300 the same overlap applies
 * between HBM and L2.  A decode pass is a chain of GEMV launches, each
 * reading the previous one's output.  Each launch's CTAs stay on their SMs
 * until their last rows are summed, and the next launch's copies cannot
 * start until those SMs free up, so HBM idles at every launch boundary.
 * Weights do not depend on earlier results.  So once every CTA of this
 * call's last launch has requested its own weight tiles, it asks L2 to fetch
 * its share of the given byte ranges (normally the leading rows of the next
 * call's codes and steps).  The next call then finds them in L2.
 *
 * Arguments, layouts, results and errors are those of w4a16_gemv (the same
 * bits for the same inputs); the ranges change timing only.
 *
 * ranges    host array of n_ranges {ptr, bytes} (read during the call, not
 *           kept).  ptr is a device address, 16-byte aligned (W4_ERR_ALIGN);
 *           a range of 0 bytes may have a NULL ptr.  Bytes past the last
 *           multiple of 16 of a range are not fetched.  The ranges are only
 *           read by L2 prefetches, never written, and must stay allocated
 *           until the call's kernels have finished.
 * n_ranges  0 .. W4_MAX_L2_RANGES (0: exactly w4a16_gemv).
 *
 * Size the ranges so that they still fit L2 together with what the next
 * call reads first.  Prefetched lines that are evicted before use are read
 * from HBM again.  Prompt chunks (M > 32, one launch of the prompt GEMM)
 * take no prefetch.
 */
#define W4_MAX_L2_RANGES 4
typedef struct w4_l2_range {
    const void *ptr;
    size_t bytes;
} w4_l2_range;

w4_status w4a16_gemv_prefetch_l2(void *y, const void *qw, const void *st, const void *x,
                                 int M, int N, int K, void *workspace, size_t workspace_bytes,
                                 int32_t *status_dev, unsigned flags,
                                 const w4_l2_range *ranges, int n_ranges, w4_stream_t stream);

/*
 * w4a16_gemv_static_scratch — w4a16_gemv without a caller-provided workspace.
 *
 * No passage of the source pages corresponds to this call; it exists for
 * callers that cannot allocate device memory: code that runs inside a host
 * framework owning every device allocation, code on a latency-critical path
 * where an allocation (which may synchronise the device) is not allowed, and
 * plain C callers with no way to keep a per-call workspace alive.  The
 * split-K scratch that w4a16_gemv takes as `workspace` is instead a fixed
 * array of W4_STATIC_SCRATCH_BYTES compiled into the library; every GPU that
 * loads the library holds it until the process exits.
 *
 * Arguments, layouts, results and errors are those of w4a16_gemv (the same
 * bits for the same inputs).  Inputs and outputs are still caller-owned
 * device buffers; the call allocates nothing (no cudaMalloc / cudaFree and
 * no allocating library routine).
 *
 *  - A shape whose split-K plan needs more than W4_STATIC_SCRATCH_BYTES of
 *    scratch (w4a16_gemv_workspace_bytes(M, N, K)) returns W4_ERR_WORKSPACE
 *    before any work is enqueued.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls on a device share that device's one array, which keeps the
 *    last call's contents: each call first clears, on its stream, the part
 *    that must start at zero.  Calls on the same device that may overlap on
 *    the GPU (for example issued to different streams) race on the array:
 *    issue them one after another in one stream per device.
 *  - W4_FLAG_PDL is accepted, but a launch that uses the array follows the
 *    clearing memset in its stream, so it does not overlap the kernel
 *    before it; launches of shapes that need no scratch overlap as with
 *    w4a16_gemv.
 */
#define W4_STATIC_SCRATCH_BYTES (256u << 10)

w4_status w4a16_gemv_static_scratch(void *y, const void *qw, const void *st, const void *x,
                                    int M, int N, int K, int32_t *status_dev,
                                    unsigned flags, w4_stream_t stream);

/*
 * w4a16_gemv_id — routed-expert GEMV through an expert (or slot) index.
 *
 * Page "Running a 26B MoE on an 8 GB Jetson by streaming experts from SSD",
 * section "Streaming without touching a single GPU kernel": the expert matmul
 * takes the expert weight tensor and a small tensor of selected ids and reads
 * expert `id` at base + id * stride, so pointing base at a pool of slots and
 * passing slot ids gives exactly the bytes, and the results, of the full
 * expert tensor.
 *
 *   e = ids[i];  W_e at qw_base + e*qw_stride_bytes, st_base + e*st_stride_bytes
 *   y[i][n] = bf16( sum_k W_e[n][k] * x[x_rows == 1 ? 0 : i][k] )
 *
 * y              bf16 [n_ids][N].
 * qw_base        uint32 [num_experts] x [N][K/8] at a stride of qw_stride_bytes
 *                (16-byte aligned base, stride a multiple of 16 and at least
 *                N*K/2).
 * st_base        bf16 steps, same rules with st_stride_bytes >= N*K/16.
 * num_experts    number of experts (or slots) behind base; ids[i] must lie
 *                in [0, num_experts).  An id outside it leaves y[i] unwritten
 *                and records W4_ERR_INDEX in *status_dev.
 * ids            device int32 [n_ids]; repeats are allowed.
 * n_ids          >= 1.
 * x              bf16 [x_rows][K], 16-byte aligned; x_rows is 1 (one row
 *                shared by every id) or n_ids (row i goes with ids[i]).
 * N, K           as for w4a16_gemv.
 */
w4_status w4a16_gemv_id(void *y, const void *qw_base, size_t qw_stride_bytes,
                        const void *st_base, size_t st_stride_bytes, int num_experts,
                        const int32_t *ids, int n_ids, const void *x, int x_rows,
                        int N, int K, int32_t *status_dev, unsigned flags,
                        w4_stream_t stream);

/*
 * w4a16_gemv_id_scaled — routed-expert GEMV whose outputs also take
 * per-expert vectors indexed by the REAL expert id.
 *
 * Page "Running a 26B MoE on an 8 GB Jetson by streaming experts from SSD",
 * section "Streaming without touching a single GPU kernel": the router's
 * choice is read by more than the expert matmul.  Per-expert scale vectors
 * and biases keep a row for every expert in memory at all times, so their
 * row must be chosen by the true expert number; only the matmul may be sent
 * to a slot pool.  Handing those tables slot numbers raises no error, it
 * just picks the wrong rows.  This call therefore takes both kinds of id,
 * and given the pool's slot table it checks on the device that every slot
 * holds the expert named for it.
 *
 *   s = ids[i] (slot, or expert, whose weights are read),  e = expert_ids[i]
 *   acc = the fp32 sum of w4a16_gemv_id for row i (same bits)
 *   y[i][n] = bf16( fma(acc, scale[e][n], bias[e][n]) )   (one fp32 rounding,
 *             then one bf16 rounding; scale 1 and bias 0 when NULL, which
 *             gives exactly the bits of w4a16_gemv_id)
 *
 * y, qw_base, qw_stride_bytes, st_base, st_stride_bytes, num_slots, ids,
 * n_ids, x, x_rows, N, K
 *                as for w4a16_gemv_id (num_slots in the role of num_experts).
 * expert_ids     device int32 [n_ids]: the real expert of row i, in
 *                [0, num_experts); outside it y[i] is left unwritten and
 *                W4_ERR_INDEX is recorded.
 * num_experts    >= 1, rows of scale and bias.
 * slot_expert    device int32 [num_slots] or NULL: the expert each slot
 *                holds (-1: none), as kept by w4_slot_pool_stage.  When
 *                given, a row with slot_expert[ids[i]] != expert_ids[i] is
 *                left unwritten and W4_ERR_OWNER is recorded.
 * scale, bias    bf16 [num_experts][N] (2-byte aligned), or NULL.
 * flags          W4_FLAG_PDL or 0.
 */
w4_status w4a16_gemv_id_scaled(void *y, const void *qw_base, size_t qw_stride_bytes,
                               const void *st_base, size_t st_stride_bytes, int num_slots,
                               const int32_t *ids, int n_ids, const void *x, int x_rows,
                               int N, int K, const int32_t *expert_ids, int num_experts,
                               const int32_t *slot_expert, const void *scale,
                               const void *bias, int32_t *status_dev, unsigned flags,
                               w4_stream_t stream);

/*
 * w4_embed_gather — dequantised rows of a 4-bit vocabulary table.
 *
 * Page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 2 — Keep the
 * Vocabulary Tables in 4-Bit": embed_tokens (which is also the output layer)
 * and the per-layer input table stay in 4-bit with a 16-bit step per group,
 * and the lookup by token id runs on the GPU; one copy of the tied table
 * serves the lookup and the output GEMV (pass the same qw/st to w4a16_gemv).
 *
 *   out[t][k] = bf16( (code[ids[t]][k] - 8) * st[ids[t]][k/32] )   (exact
 *   product, one rounding)
 *
 * out        bf16 [T][K], 16-byte aligned.
 * qw, st     the table, layout as for w4a16_gemv with N = V rows, 16-byte
 *            aligned.
 * ids        device int32 [T]; an id outside [0, V) leaves out[t] unwritten
 *            and records W4_ERR_INDEX.
 * T, V       >= 1.  K as for w4a16_gemv.
 */
w4_status w4_embed_gather(void *out, const void *qw, const void *st, const int32_t *ids,
                          int T, int V, int K, int32_t *status_dev, unsigned flags,
                          w4_stream_t stream);

/*
 * w4_pack — pack 4-bit codes into the qw layout.
 *
 * codes      device uint8 [N][K], values 0..15.  A larger value records
 *            W4_ERR_VALUE and leaves that word of qw unwritten.
 * qw         device uint32 [N][K/8], 16-byte aligned.
 * K          multiple of 32.
 */
w4_status w4_pack(void *qw, const uint8_t *codes, int N, int K, int32_t *status_dev,
                  w4_stream_t stream);

/*
 * w4_quantize — quantise fp32 weights into (qw, st).
 *
 * Page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 2 — Keep the
 * Vocabulary Tables in 4-Bit" says only that each group's step is recovered
 * from its 4-bit grid.  This helper uses the plain signed-absmax rule, per
 * group of 32 along K:
 *   m    = element of largest |w| (the first in K order on ties)
 *   step = bf16(m / -8)                     (nearest even)
 *   code = 8 if step == 0, else clamp(rint(w / step) + 8, 0, 15)
 *          with IEEE fp32 division and rint rounding half to even,
 * so the element m becomes code 0 and dequantises back to m.
 *
 * w          device fp32 [N][K], finite values, 16-byte aligned.
 * qw, st     outputs as for w4a16_gemv, 16-byte aligned.
 */
w4_status w4_quantize(void *qw, void *st, const float *w, int N, int K, w4_stream_t stream);

/*
 * Expert slot pool (host side of the routed-expert path).
 *
 * Page "Running a 26B MoE on an 8 GB Jetson by streaming experts from SSD",
 * section "Streaming without touching a single GPU kernel": each MoE layer
 * keeps a persistent pool of expert-sized slots and a small slot-id tensor;
 * for every token an LFU cache finds which requested experts are resident,
 * loads the misses into their assigned slots, and writes the slot indices for
 * the expert matmul.  Policy (the page leaves the details open): every
 * request counts as one use; misses take the lowest free slot, else evict the
 * resident expert not requested now with the fewest uses, then the least
 * recently used, then the lowest slot index; misses are placed in request
 * order; a repeated id shares one slot.
 *
 * Only the expert matmul may see slot ids; anything else indexed by expert
 * (per-expert scales, biases, adapters) must keep the real ids.
 */
typedef struct w4_slot_pool w4_slot_pool;

/* Create a pool for num_experts experts and num_slots slots (host memory). */
w4_status w4_slot_pool_create(w4_slot_pool **pool, int num_experts, int num_slots);
void w4_slot_pool_destroy(w4_slot_pool *pool);

/*
 * Host-only remap of one request of k expert ids (host int32 [k]).
 * Writes slot_ids (host int32 [k]) and the misses as parallel arrays
 * miss_experts / miss_slots (host int32 [k] each, *n_miss entries).
 * Returns W4_ERR_INDEX for an id outside [0, num_experts) and W4_ERR_STATE
 * when k names more distinct experts than there are slots; the pool is then
 * unchanged.
 */
w4_status w4_slot_pool_remap(w4_slot_pool *pool, const int32_t *expert_ids, int k,
                             int32_t *slot_ids, int32_t *miss_experts, int32_t *miss_slots,
                             int *n_miss);

/*
 * Remap one request and stage it on `stream`: each missed expert's codes
 * (qw_expert_bytes from full_qw + e*qw_stride to pool_qw + s*qw_stride) and
 * steps (likewise with st_*) are copied into its slot and the k slot ids are
 * written into slot_ids_dev (device int32 [k], k <= 64).  When every pointer,
 * stride and size is a multiple of 16 bytes, one kernel launch does all of
 * it; otherwise one cudaMemcpyAsync per copy, then a tiny kernel for the ids.
 * If any of it fails to enqueue, the experts of this request that were being
 * loaded are dropped from the pool (their slots become free) and
 * W4_ERR_STATE is returned, so stale slot contents are never used.
 * slot_ids / n_miss (host, optional, may be NULL) receive the remap.
 *
 * full_qw / full_st may live in device memory or in page-locked host memory
 * (on GB300 the Grace CPU's memory, read by the GPU over NVLink-C2C): the
 * fill kernel reads them in place, the copy fallback uses cudaMemcpyDefault.
 *
 * slot_expert_dev (device int32 [num_slots], or NULL) is the pool's slot
 * table for w4a16_gemv_id_scaled: the caller fills it with -1 once, then each
 * stage marks the slots it refills as holding no expert before their copies
 * and names the new expert once they are complete, in stream order.
 */
w4_status w4_slot_pool_stage(w4_slot_pool *pool, const int32_t *expert_ids, int k,
                             void *pool_qw, const void *full_qw, size_t qw_stride_bytes,
                             size_t qw_expert_bytes, void *pool_st, const void *full_st,
                             size_t st_stride_bytes, size_t st_expert_bytes,
                             int32_t *slot_ids_dev, int32_t *slot_expert_dev,
                             int32_t *slot_ids, int *n_miss, w4_stream_t stream);

/*
 * Device-side slot pool: the same policy decided on the GPU, so a routed step
 * (router ids on the device -> remap -> fills -> w4a16_gemv_id) needs no host
 * round trip and can be captured in a CUDA graph.  The pool's whole state
 * lives in a caller-owned device buffer of w4_dev_pool_state_bytes bytes
 * (16-byte aligned), set up once with w4_dev_pool_init.  num_slots <= 64 and
 * <= num_experts <= 3980.
 */
size_t w4_dev_pool_state_bytes(int num_experts, int num_slots);

/* Reset the state on `stream`: every slot free, every count 0. */
w4_status w4_dev_pool_init(void *state, int num_experts, int num_slots, w4_stream_t stream);

/*
 * Enqueue the remap of the k (<= 64) device int32 expert ids at `ids` and the
 * fills of the misses: one single-thread kernel decides, one kernel copies
 * each missed expert's codes and steps (as w4_slot_pool_stage, every
 * pointer, stride and size a multiple of 16 bytes; sources in device memory
 * or page-locked host memory) and names the new experts in the slot table
 * (slot_expert_dev, optional, the caller fills it with -1 once).  The slot
 * ids go to slot_ids_dev.  A request with an id outside [0, num_experts) or
 * more distinct ids than slots changes nothing, writes -1 slot ids (the
 * routed GEMV then leaves those rows unwritten) and records W4_ERR_INDEX or
 * W4_ERR_STATE in *status_dev.  W4_FLAG_PDL: the remap waits for earlier
 * kernels (the router) only where it reads the ids.
 */
w4_status w4_dev_pool_stage(void *state, int num_experts, int num_slots, const int32_t *ids,
                            int k, void *pool_qw, const void *full_qw, size_t qw_stride_bytes,
                            size_t qw_expert_bytes, void *pool_st, const void *full_st,
                            size_t st_stride_bytes, size_t st_expert_bytes,
                            int32_t *slot_ids_dev, int32_t *slot_expert_dev,
                            int32_t *status_dev, unsigned flags, w4_stream_t stream);

/* Counters of a device-side pool (synchronous device-to-host read). */
w4_status w4_dev_pool_stats(const void *state, int num_experts, int num_slots,
                            long long *requests, long long *hits, long long *misses);

/* Counters since creation: requests served (ids), hits, misses (copies). */
void w4_slot_pool_stats(const w4_slot_pool *pool, long long *requests, long long *hits,
                        long long *misses);

/*
 * Launch plan chosen for a w4a16_gemv shape (for tests and benchmarks).
 * Returns W4_OK and fills *info, or an argument error for an invalid shape.
 */
typedef struct w4_plan_info {
    int path;           /* 1 = tile-streamed CUDA-core packed-fp16 kernel,
                           2 = tensor-core small-batch kernel (up to 32 rows
                           per launch), 3 = tensor-core prompt GEMM (33 to
                           256 rows in one launch) */
    int ctas;           /* CTAs launched */
    int slices;         /* K slices (split-K); 1 = none */
    int threads;        /* threads per CTA (7 consumer warps + 1 copy warp) */
    int team;           /* lanes that share one output row */
    int unit_rows;      /* output rows of one streamed tile */
    int chunk_groups;   /* 32-code groups per K chunk of the row reduction */
    int rows_per_lane;  /* rows a lane works on together (activation reuse) */
    int smem_bytes;     /* dynamic shared memory per CTA */
    int rows_per_call;  /* activation rows handled per launch */
    int chunk_steps;    /* groups per lane per K chunk */
    int stages;         /* shared-memory tiles in flight per CTA */
    int ctas_per_sm;    /* resident CTAs per SM the plan is sized for */
    int tmpl_team;      /* team size compiled into the kernel (0: generic) */
    int tmpl_chunk;     /* chunk steps compiled into the kernel (0: generic) */
    int dynamic_windows; /* path 1: CTAs take windows of unit_rows rows from a
                            counter at run time (dense calls with many windows per
                            CTA, and routed calls with many windows, within one id
                            each).  path 2: balanced runs, each CTA an equal share
                            of the (128-row tile, 256-code slice) work; a tile cut
                            between two CTAs hands its rows' running sums over
                            through the workspace (taken only when the call's
                            workspace is w4a16_gemv_workspace_bytes large) */
} w4_plan_info;

w4_status w4a16_gemv_plan(int M, int N, int K, w4_plan_info *info);

/* The plan of a w4a16_gemv call with the given flags (a pinned path plans
 * that path's launch).  W4_ERR_SHAPE when the pinned path cannot run K. */
w4_status w4a16_gemv_plan_flags(int M, int N, int K, unsigned flags, w4_plan_info *info);

/* The same for a w4a16_gemv_id call with n_ids ids and x_rows activation
 * rows (path is always 1). */
w4_status w4a16_gemv_id_plan(int n_ids, int x_rows, int N, int K, w4_plan_info *info);

/*
 * w4a16_gemv_chain — a list of W4A16 GEMVs in one launch.
 *
 * Page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 3 — Multiply
 * Straight From the Packed Weights": a decoded token is the product of an
 * activation vector with each weight matrix in turn, and its rate is set by
 * how fast the packed words stream from memory.  This call runs a whole list
 * of such products ("tasks": the projections of a decode pass, or a routed
 * layer's gate/up then down product, page "Running a 26B MoE on an 8 GB
 * Jetson by streaming experts from SSD", section "Streaming without touching
 * a single GPU kernel") as one persistent launch, one CTA per SM, whose
 * weight stream does not pause between tasks (the copy warp keeps fetching
 * later tasks' weights while the products wait for their inputs).
 *
 * Task j computes, with the arithmetic of the same call made alone:
 *   dense  (ids == NULL): y[N] = W x                     (w4a16_gemv, M = 1)
 *   routed (ids != NULL): y[i][N] = W_{ids[i]} x_i       (w4a16_gemv_id), for
 *          i < n_ids, expert e at qw + e * qw_stride, st + e * st_stride,
 *          x_i = row i of x when x_rows == n_ids > 1, else row 0;
 * with W4_TASK_SILU_MUL each activation row is [gate K | up K] and the
 * product takes silu(gate) * up (as W4_FLAG_SILU_MUL).  Every task's outputs
 * are bitwise those of the single call (tested).
 *
 * Order and dependencies: `dep` names an earlier task (index < j) whose
 * outputs task j reads (its x), or -1.  Task j's products start only after
 * every output of task `dep` is written; weights of later tasks may already
 * stream meanwhile.  When both tasks are routed on the same ids, task j's
 * activation rows are `dep`'s output (x == dep's y, x_rows == n_ids, a row
 * of K, or 2K gated, values == dep's N), expert i of task j waits only for
 * expert i of `dep` (a routed layer's down product after its gate/up).  A task with dep = -1 must find its x ready when the
 * launch starts.  For a strict sequence (each projection reading the one
 * before, as a decoder does) set dep = j - 1.  Outputs of tasks are written
 * in an unspecified order; a task must not write what another task of the
 * launch reads, except through `dep`.
 *
 * Arguments, layouts and alignment of each task are those of w4a16_gemv /
 * w4a16_gemv_id (K multiple of 32 up to W4_MAX_K, qw / st / x 16-byte
 * aligned, y 2-byte aligned, expert strides multiples of 16 and at least one
 * expert).  n_tasks <= W4_CHAIN_MAX_TASKS (the task list travels in the
 * launch's parameters, so a CUDA graph that captures the call keeps it).
 *
 * workspace: caller-owned device memory of
 * w4a16_gemv_chain_workspace_bytes(tasks, n_tasks) bytes (16-byte aligned), zeroed
 * before the first call; each launch re-arms it when it completes.  After a
 * call that reported a device-side error, zero it again.  Calls that share a
 * workspace must not overlap on the GPU.
 *
 * Errors: host-detectable ones return before any launch (W4_ERR_ARG for a
 * null pointer, an unknown flag, N < 1 or a `dep` that is not an earlier
 * task; W4_ERR_SHAPE / W4_ERR_ALIGN as for the single calls, or when the
 * tasks' activation rows and the smallest stages do not fit shared memory;
 * W4_ERR_WORKSPACE).  Device-side: an expert id out of range leaves that
 * item's rows unwritten and records W4_ERR_INDEX; a wait that exceeds about
 * a second (a dependency that never completes) records W4_ERR_TIMEOUT.
 * flags: W4_FLAG_PDL.
 */
#define W4_CHAIN_MAX_TASKS 320
#define W4_TASK_SILU_MUL 1u   /* task: x rows are [gate K | up K] -> silu(gate) * up */

typedef struct w4_gemv_task {
    void *y;                  /* bf16 [N] (dense) or [n_ids][N] (routed) */
    const void *qw;           /* packed codes: the matrix, or expert 0 of a routed task */
    const void *st;           /* bf16 steps, likewise */
    const void *x;            /* bf16 activation row(s) */
    const int32_t *ids;       /* routed: n_ids expert (or slot) ids on the device; NULL: dense */
    size_t qw_stride;         /* routed: bytes between experts' codes */
    size_t st_stride;         /* routed: bytes between experts' steps */
    int num_experts;          /* routed: valid ids are 0 .. num_experts - 1 */
    int n_ids;                /* routed: output rows of y; ignored for dense tasks */
    int x_rows;               /* routed: 1 (shared row) or n_ids */
    int N, K;
    int dep;                  /* earlier task whose outputs this one reads, or -1 */
    unsigned flags;           /* W4_TASK_SILU_MUL */
} w4_gemv_task;

/* Workspace of a chain: two ints plus one per task (one per id of a routed
 * task), rounded up to 256 bytes; 0 for an invalid task list. */
size_t w4a16_gemv_chain_workspace_bytes(const w4_gemv_task *tasks, int n_tasks);

w4_status w4a16_gemv_chain(const w4_gemv_task *tasks, int n_tasks, void *workspace,
                           size_t workspace_bytes, int32_t *status_dev, unsigned flags,
                           w4_stream_t stream);

/* Launch shape of a chain (planned for the current device, or for GB300
 * figures without one): CTAs and threads, the dot instantiation (0: hidden
 * 5376 / intermediate 21504, 1: 2048 / 8192, 2: routed 2816 / 704,
 * 3: generic), stages and their size, shared memory, windows in all. */
typedef struct w4_chain_plan_info {
    int ctas, threads, instantiation, stages, stage_bytes, smem_bytes, windows;
} w4_chain_plan_info;

w4_status w4a16_gemv_chain_plan(const w4_gemv_task *tasks, int n_tasks, w4_chain_plan_info *info);

/* Window shape of one task of a chain: rows per window, rows per lane, lane
 * team, groups per lane per chunk, chunks per row, windows per item, and
 * which of the instantiation's two dot loops (0, 1) runs it. */
typedef struct w4_chain_task_info {
    int rows_per_window, rows_per_lane, team, chunk_steps, chunks, windows_per_item, dot;
} w4_chain_task_info;

w4_status w4a16_gemv_chain_task_plan(const w4_gemv_task *tasks, int n_tasks, int task,
                                     w4_chain_task_info *info);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */

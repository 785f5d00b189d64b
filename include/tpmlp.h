/*
 * tpmlp - the Megatron tensor-parallel Transformer MLP block on one GB300
 * (sm_103a), with all p shards on one device.
 *
 * The block (sources are web pages on Megatron tensor parallelism):
 *   - column-parallel first layer: A [h, f] is split along its output columns
 *     into p shards A_i [h, f/p]; every shard sees the whole input X and
 *     computes H_i = X A_i + b1_i, Y_i = GeLU(H_i) with no communication
 *     ("列并行" article, sections 切分原理 / 数学基础 / MLP 应用;
 *      "Megatron 专家面试题 Level 2", M025);
 *   - row-parallel second layer: B [f, h] is split along its input rows into
 *     B_i [f/p, h]; shard i computes the full-shape partial Z_i = Y_i B_i and
 *     the block returns Z = sum_i Z_i + b2 (Level 2, M026 and M027;
 *     "分布式并行训练全景", 考点 2).  The pages place that sum in an
 *     All-Reduce; here it is the row GEMM's own K loop, accumulated in fp32
 *     tensor memory across all shards, followed by one bf16 store;
 *   - backward: dA_i = X^T dH_i and dB_i = Y_i^T dZ stay local, dX is the sum
 *     of the shard contributions dH_i A_i^T (Level 2, M025 追问 and M026).
 *
 * Conventions shared by every entry point
 *   Layout.  Activations are [s, b, h] row-major; token (s_idx, b_idx) is row
 *     m = s_idx * b + b_idx of an [M, h] matrix, M = s * b.  Shard tensors are
 *     stored shard-contiguous: A_sh [p][h][f/p], B_sh [p][f/p][h] (the same
 *     bytes as B [f, h] row-major), b1_sh [p][f/p] (the same bytes as b1 [f]),
 *     Y_sh / H_sh / dH [p][M][f/p].  All matrices are row-major.
 *   Memory.  Every pointer is caller-owned device memory (for example
 *     allocated by PyTorch).  The library never allocates device memory,
 *     frees or synchronises inside these calls, and creates no streams or
 *     events: every kernel of a call goes to `stream`, or to a side stream the
 *     caller has registered (tpmlp_set_side_stream).  Workspaces are passed
 *     in with the sizes stated.  Calls are stream ordered and asynchronous: they return after
 *     the kernels are enqueued on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  The GEMM kernels are launched with programmatic
 *     dependent launch: their set-up may overlap the end of the preceding
 *     kernel in the stream, but they touch no global memory before that
 *     kernel has completed, so stream order holds as for any launch.
 *   Validation.  Arguments are checked on the host before anything is
 *     enqueued, in this order: NULL pointers (TPMLP_ERR_NULL), shapes
 *     (TPMLP_ERR_SHAPE: s, b >= 0; h, ffn, p >= 1; sizes below 2^31 rows),
 *     divisibility (TPMLP_ERR_DIVISIBILITY: ffn % p, and h % p where stated),
 *     dtype (TPMLP_ERR_DTYPE), alignment (TPMLP_ERR_ALIGNMENT: every pointer
 *     16-byte aligned and every row pitch a multiple of 16 bytes, i.e. h and
 *     ffn/p multiples of 8 for bf16, of 4 for fp32), aliasing
 *     (TPMLP_ERR_ALIAS: no output overlaps an input or another output), then
 *     the device (TPMLP_ERR_ARCH unless compute capability 10.3).  An empty
 *     batch (s * b == 0) is valid and enqueues nothing.  There is no CPU
 *     fallback.
 *   Errors.  A failed launch returns TPMLP_ERR_CUDA.  Kernels never trap: a
 *     device-side wait that runs past its time limit records a status word
 *     and returns; tpmlp_device_status() reports it as TPMLP_ERR_TIMEOUT.
 *     tpmlp_last_error() gives a thread-local message for the last failure.
 *   Numerics.  bf16 inputs, fp32 accumulation in tensor memory, bf16 outputs
 *     (rounded to nearest even); fp32 inputs run on fp32 FMA (no TF32).
 */
#ifndef TPMLP_H
#define TPMLP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TPMLP_OK = 0,
    TPMLP_ERR_NULL = 1,
    TPMLP_ERR_SHAPE = 2,
    TPMLP_ERR_DIVISIBILITY = 3,
    TPMLP_ERR_DTYPE = 4,
    TPMLP_ERR_ALIGNMENT = 5,
    TPMLP_ERR_ALIAS = 6,
    TPMLP_ERR_ARCH = 7,
    TPMLP_ERR_CUDA = 8,
    TPMLP_ERR_TIMEOUT = 9,
    TPMLP_ERR_DEVICE = 10
} tpmlp_status;

typedef enum { TPMLP_BF16 = 0, TPMLP_F32 = 1 } tpmlp_dtype;

typedef enum { TPMLP_ACT_NONE = 0, TPMLP_ACT_GELU_ERF = 1 } tpmlp_act;

/*
 * Column-parallel layer for all p shards in one launch
 * ("列并行" article, 数学基础 and MLP 应用; Level 2, M025):
 *   H_i = X A_i + b1_i,   Y_i = act(H_i),   act = GeLU(z) = z * Phi(z) (erf form) or identity.
 *   X     [M, h]            dt
 *   A_sh  [p][h][ffn/p]     dt
 *   b1_sh [p][ffn/p]        dt, may be NULL (no bias)
 *   Y_sh  [p][M][ffn/p]     dt, output
 *   H_sh  [p][M][ffn/p]     dt, optional output of the pre-activation (NULL = not saved)
 * Requires ffn % p == 0.
 */
tpmlp_status tpmlp_column_fwd(const void* X, const void* A_sh, const void* b1_sh, void* Y_sh, void* H_sh,
                              int64_t s, int64_t b, int64_t h, int64_t ffn, int p,
                              tpmlp_dtype dt, tpmlp_act act, void* stream);

/*
 * Row-parallel layer with the shard sum on device
 * (Level 2, M026; "分布式并行训练全景", 考点 2: Z = Z_1 + Z_2 + ...):
 *   Z = sum_i Y_i B_i + b2     (b2 added once, after the sum)
 *   Y_sh [p][M][ffn/p] dt;  B_sh [p][ffn/p][h] dt;  b2 [h] dt or NULL;  Z [M, h] dt, output.
 * Requires ffn % p == 0.
 */
tpmlp_status tpmlp_row_fwd(const void* Y_sh, const void* B_sh, const void* b2, void* Z,
                           int64_t s, int64_t b, int64_t h, int64_t ffn, int p,
                           tpmlp_dtype dt, void* stream);

/*
 * The MLP block forward: column (GeLU, erf form) then row, as two launches
 * ("列并行" article, MLP 应用: no gather between the layers, one sum at the end).
 *   Y_ws  [p][M][ffn/p] dt  caller workspace, holds Y on return (needed by the backward)
 *   H_sh  [p][M][ffn/p] dt  optional pre-activation save for the backward (NULL = not saved)
 *   other arguments as in tpmlp_column_fwd / tpmlp_row_fwd.
 * Requires ffn % p == 0 and h % p == 0.
 */
tpmlp_status tpmlp_mlp_fwd(const void* X, const void* A_sh, const void* b1_sh, const void* B_sh, const void* b2,
                           void* Z, void* Y_ws, void* H_sh,
                           int64_t s, int64_t b, int64_t h, int64_t ffn, int p,
                           tpmlp_dtype dt, void* stream);

/*
 * The MLP block backward from dZ (Level 2, M025 追问 and M026; chain rule):
 *   dY_i = dZ B_i^T,  dH_i = dY_i * GeLU'(H_i),  GeLU'(z) = Phi(z) + z phi(z)
 *   dB_i = Y_i^T dZ,  dA_i = X^T dH_i,  db1_i = 1^T dH_i,  db2 = 1^T dZ   (local)
 *   dX   = sum_i dH_i A_i^T                                                (summed on device)
 * Inputs:  X [M,h], A_sh, B_sh, H_sh and Y_sh from the forward, dZ [M,h]   (all dt)
 * Outputs: dX [M,h] dt;  dA_sh [p][h][ffn/p], dB_sh [p][ffn/p][h], db1_sh [p][ffn/p] (or NULL),
 *          db2 [h] (or NULL), all grad_dt (fp32 recommended for bf16 inputs).
 * Workspace: dH_ws [p][M][ffn/p] dt, holds dH on return.
 * Requires ffn % p == 0 and h % p == 0; grad_dt must be TPMLP_F32 when dt is TPMLP_F32.
 * Launch order on `stream`: dH, dB, db2, db1, dA, dX (where a side stream of the caller's is
 * registered, the GEMMs or the column sums may run beside one another: tpmlp_set_side_stream).
 */
tpmlp_status tpmlp_mlp_bwd(const void* X, const void* A_sh, const void* B_sh, const void* H_sh, const void* Y_sh,
                           const void* dZ, void* dX, void* dA_sh, void* dB_sh, void* db1_sh, void* db2,
                           void* dH_ws, int64_t s, int64_t b, int64_t h, int64_t ffn, int p,
                           tpmlp_dtype dt, tpmlp_dtype grad_dt, void* stream);

/*
 * The block with its shards spread over several GPUs: what one rank computes
 * ("分布式并行训练全景", 考点 2: each card holds a column slice A_i of the first
 * weight and the matching row slice B_i of the second, computes GeLU(X A_i) B_i
 * with no exchange in between, and one All-Reduce sums the partials; Level 2,
 * M025 追问: in the backward the weight gradients stay local and the dX
 * contributions are summed by an All-Reduce; M027: the sum comes once, at the
 * end of the block).  The exchange itself is the caller's (NCCL or any other
 * collective); these calls compute the rank-local parts on this GPU and the
 * step after the sum.
 *
 * tpmlp_mlp_fwd_partial: this rank's p local shards (its slice of A's columns,
 * b1 and B's rows, laid out as in tpmlp_mlp_fwd with ffn = the rank's FFN width)
 *   H_i = X A_i + b1_i,  Y_i = GeLU(H_i),  Z_part = sum_{local i} Y_i B_i
 *   Z_part [M, h] fp32 output (no b2: it is added once, after the All-Reduce,
 *   by tpmlp_sum_finish); Y_ws, H_sh and the requirements as in tpmlp_mlp_fwd.
 *   With every shard on one rank, Z = round(Z_part + b2) is tpmlp_mlp_fwd's
 *   result up to the fp32 summation order.
 */
tpmlp_status tpmlp_mlp_fwd_partial(const void* X, const void* A_sh, const void* b1_sh, const void* B_sh,
                                   float* Z_part, void* Y_ws, void* H_sh,
                                   int64_t s, int64_t b, int64_t h, int64_t ffn, int p,
                                   tpmlp_dtype dt, void* stream);

/*
 * tpmlp_mlp_bwd_partial: the rank-local backward.  As tpmlp_mlp_bwd on this
 * rank's shards (dH, dA_i, dB_i, db1_i all local; db2 = 1^T dZ needs only the
 * replicated dZ, so every rank gets the whole of it), except that dX_part
 * [M, h] fp32 receives this rank's contribution sum_{local i} dH_i A_i^T, to be
 * summed over the ranks by the caller's All-Reduce and rounded by
 * tpmlp_sum_finish (bias NULL).  Launch order on `stream`: dH, dB, db2, db1,
 * dA, dX_part (the sums on a registered side stream as in tpmlp_mlp_bwd).
 */
tpmlp_status tpmlp_mlp_bwd_partial(const void* X, const void* A_sh, const void* B_sh, const void* H_sh,
                                   const void* Y_sh, const void* dZ, float* dX_part, void* dA_sh, void* dB_sh,
                                   void* db1_sh, void* db2, void* dH_ws, int64_t s, int64_t b, int64_t h,
                                   int64_t ffn, int p, tpmlp_dtype dt, tpmlp_dtype grad_dt, void* stream);

/*
 * The step after the All-Reduce of fp32 partial sums (考点 2; M026: b2 is added
 * once, to the sum, never per rank):
 *   out[r][c] = round_dt(S[r][c] + bias[c])
 *   S [rows, cols] fp32 (the summed partials), bias [cols] dt or NULL,
 *   out [rows, cols] dt (bf16: rounded to nearest even; fp32: the sum itself).
 * cols must be a multiple of 8 (bf16) or 4 (fp32); out must not overlap S or bias.
 */
tpmlp_status tpmlp_sum_finish(const float* S, const void* bias, void* out, int64_t rows, int64_t cols,
                              tpmlp_dtype dt, void* stream);

/*
 * Row-parallel layer backward (Level 2, M026: the row layer's input gradient is
 * naturally the input shard; its weight gradient is local):
 *   dY_i = dZ B_i^T            act = NONE
 *   dY_i = (dZ B_i^T) * GeLU'(H_i)   act = GELU_ERF: the gradient at the column
 *                                     layer's pre-activation, GeLU'(z) = Phi(z) + z phi(z)
 *   dB_i = Y_i^T dZ,  db2 = 1^T dZ (optional)
 * Inputs:  Y_sh [p][M][ffn/p] (this layer's input), B_sh [p][ffn/p][h], dZ [M,h] (dt);
 *          H_sh [p][M][ffn/p] (dt; required iff act = GELU_ERF, else ignored).
 * Outputs: dY_sh [p][M][ffn/p] dt;  dB_sh [p][ffn/p][h] and db2 [h] (or NULL) grad_dt.
 * Requires ffn % p == 0; grad_dt must be TPMLP_F32 when dt is TPMLP_F32.
 */
tpmlp_status tpmlp_row_bwd(const void* Y_sh, const void* B_sh, const void* dZ, const void* H_sh, void* dY_sh,
                           void* dB_sh, void* db2, int64_t s, int64_t b, int64_t h, int64_t ffn, int p,
                           tpmlp_dtype dt, tpmlp_dtype grad_dt, tpmlp_act act, void* stream);

/*
 * Column-parallel layer backward (Level 2, M025 追问: dW_i = X^T dY_i is local;
 * the input-gradient contributions dY_i W_i^T of all shards are summed):
 *   dA_i = X^T dY_i,  db1_i = 1^T dY_i (optional),  dX = sum_i dY_i A_i^T (summed on device)
 * Inputs:  X [M,h], A_sh [p][h][ffn/p], dY_sh [p][M][ffn/p] (dt).
 * Outputs: dX [M,h] dt;  dA_sh [p][h][ffn/p] and db1_sh [p][ffn/p] (or NULL) grad_dt.
 * Requires ffn % p == 0; grad_dt must be TPMLP_F32 when dt is TPMLP_F32.
 * tpmlp_mlp_bwd is tpmlp_row_bwd (GeLU') followed by tpmlp_column_bwd.
 */
tpmlp_status tpmlp_column_bwd(const void* X, const void* A_sh, const void* dY_sh, void* dX, void* dA_sh,
                              void* db1_sh, int64_t s, int64_t b, int64_t h, int64_t ffn, int p,
                              tpmlp_dtype dt, tpmlp_dtype grad_dt, void* stream);

/*
 * SwiGLU variant of the block (Level 2, M027: a gated activation works on local
 * pairs of the FFN shard, so the column + row split still needs only the final sum):
 *   Hg_i = X G_i + bg_i,  Hu_i = X U_i + bu_i,  Y_i = silu(Hg_i) * Hu_i,  Z = sum_i Y_i B_i + b2,
 *   silu(x) = x / (1 + exp(-x)).
 * The gate and up weights of each shard are packed by tpmlp_swiglu_pack into
 *   W_sh [p][h][2 ffn/p]: columns 256 b .. 256 b + 127 = gate features 128 b ..,
 *                         columns 256 b + 128 .. 256 b + 255 = up features 128 b ..
 * bw_sh [p][2 ffn/p] is the packed bias (or NULL); Y_ws [p][M][ffn/p] holds Y on return;
 * H_ws [p][M][2 ffn/p] fp32 (or NULL) receives the packed pre-activations for the backward, in
 * fp32 because the backward multiplies by the up pre-activation itself (dHg = dY Hu silu'(Hg)):
 * rounding Hg and Hu to bf16 would roughly double the bf16 error of dX against the GeLU block.
 * Requires bf16, ffn % p == 0, h % p == 0 and ffn/p a multiple of 128.
 */
tpmlp_status tpmlp_swiglu_mlp_fwd(const void* X, const void* W_sh, const void* bw_sh, const void* B_sh,
                                  const void* b2, void* Z, void* Y_ws, void* H_ws, int64_t s, int64_t b, int64_t h,
                                  int64_t ffn, int p, tpmlp_dtype dt, void* stream);

/*
 * SwiGLU backward from dZ:  dY_i = dZ B_i^T,  dHg = dY Hu silu'(Hg),  dHu = dY silu(Hg),
 *   dW_i = X^T [dHg | dHu] (packed), dbw_i = 1^T [dHg | dHu], dB_i = Y_i^T dZ, db2 = 1^T dZ,
 *   dX = sum_i [dHg | dHu]_i W_i^T  (= dHg G^T + dHu U^T, summed on device).
 *   silu'(x) = sigma(x) (1 + x (1 - sigma(x))).
 * Inputs: X, W_sh, B_sh, Y_ws and dZ (bf16); H_ws (packed fp32 pre-activations from the forward).
 * Outputs: dX bf16; dW_sh [p][h][2 ffn/p], dB_sh, dbw_sh [p][2 ffn/p] (or NULL), db2 (or NULL) grad_dt.
 * Workspace: dH_ws [p][M][2 ffn/p] bf16 (holds the packed dHg, dHu on return).
 * Launch order on `stream`: the dY GEMM with the SwiGLU' epilogue, dB, db2, dbw, dW, dX (db2
 * and dbw beside dX where a side stream is registered, as in tpmlp_mlp_bwd).
 */
tpmlp_status tpmlp_swiglu_mlp_bwd(const void* X, const void* W_sh, const void* B_sh, const void* H_ws,
                                  const void* Y_ws, const void* dZ, void* dX, void* dW_sh, void* dB_sh, void* dbw_sh,
                                  void* db2, void* dH_ws, int64_t s, int64_t b, int64_t h, int64_t ffn, int p,
                                  tpmlp_dtype dt, tpmlp_dtype grad_dt, void* stream);

/*
 * SwiGLU weight packing (bit-exact): G, U [rows][ffn] -> W_sh [p][rows][2 ffn/p] as described at
 * tpmlp_swiglu_mlp_fwd (rows = 1 packs the biases); inverse != 0 unpacks W_sh into G and U.
 * Requires ffn % p == 0 and ffn/p a multiple of 128.
 */
tpmlp_status tpmlp_swiglu_pack(void* G, void* U, void* W_sh, int64_t rows, int64_t ffn, int p, tpmlp_dtype dt,
                               int inverse, void* stream);

/*
 * The MLP block forward without a caller workspace.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate device
 * memory where they run the block (for example an inference-engine plugin whose
 * host engine owns all device memory, or a runtime that forbids allocation after
 * start-up because an allocation can synchronise the device).
 *   Same arguments and results as tpmlp_mlp_fwd without Y_ws and H_sh: the
 *   intermediate Y lives in a fixed array inside the library of
 *   TPMLP_NOALLOC_SCRATCH_BYTES bytes (32 MiB), which every GPU that loads the
 *   library holds until the process exits.  Calls needing more than that
 *   (s*b*ffn*element size bytes) return TPMLP_ERR_SHAPE.
 *   This call allocates nothing (no cudaMalloc, no allocating library routine).
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make that
 *   first call before any stream capture.  Under CUDA's lazy module loading
 *   (the default) that first look-up, or the first launch of a kernel of this
 *   library, may load the library's code onto the device, and loading creates
 *   the array there: device memory that the driver takes at that moment.  A
 *   caller that must not see any allocation after start-up makes one call at
 *   start-up (or sets CUDA_MODULE_LOADING=EAGER) before its no-allocation
 *   region; later calls take no device memory.
 *   Every call shares the one array per device and it keeps the last call's
 *   contents; each call overwrites all of the Y it reads, so nothing needs
 *   clearing.  Calls whose kernels overlap on the GPU (different streams, or
 *   threads without ordering) race on the array.
 */
#define TPMLP_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
tpmlp_status tpmlp_mlp_fwd_noalloc(const void* X, const void* A_sh, const void* b1_sh, const void* B_sh,
                                   const void* b2, void* Z, int64_t s, int64_t b, int64_t h, int64_t ffn, int p,
                                   tpmlp_dtype dt, void* stream);

/*
 * Column shard layout ("列并行" article, 切分原理: W = [W(1) || ... || W(p)];
 * the article's NumPy demo uses np.split(W, p, axis=1)):
 *   W_sh[i][r][c] = W[r][i * cols/p + c],   W [rows, cols] dt,  W_sh [p][rows][cols/p] dt.
 * Requires cols % p == 0 and (cols/p) a multiple of 8 (bf16) / 4 (fp32). Bit-exact copy.
 */
tpmlp_status tpmlp_shard_columns(const void* W, void* W_sh, int64_t rows, int64_t cols, int p,
                                 tpmlp_dtype dt, void* stream);

/* The inverse of tpmlp_shard_columns: W[r][i * cols/p + c] = W_sh[i][r][c]. */
tpmlp_status tpmlp_unshard_columns(const void* W_sh, void* W, int64_t rows, int64_t cols, int p,
                                   tpmlp_dtype dt, void* stream);

/*
 * Per-head interleave of a packed QKV projection ("Tencent Hunyuan AI Infra
 * interview", answer on QKV: interleave the packed matrix so that each head's
 * Q, K and V land on the same card; Level 2, M028: QKV column parallel by heads).
 *   W_qkv [rows, 3h] = [Q | K | V] (each h wide, head g at columns g*d..g*d+d-1, d = h/n_heads)
 *   W_out [rows, 3h] head-major: dst column (3g + t) d + e = src column t h + g d + e, t in {0,1,2}.
 * After it, a p-way column split gives rank r the heads r n/p .. (r+1) n/p - 1 with their Q, K, V.
 * inverse != 0 applies the inverse permutation.  Requires n_heads % p == 0 and h % n_heads == 0.
 * Bit-exact copy.
 */
tpmlp_status tpmlp_qkv_interleave(const void* W_qkv, void* W_out, int64_t rows, int64_t h, int64_t n_heads,
                                  int p, tpmlp_dtype dt, int inverse, void* stream);

/* Host-only: the source column of destination column dst_col of tpmlp_qkv_interleave (-1 on bad args). */
int64_t tpmlp_qkv_src_col(int64_t dst_col, int64_t h, int64_t n_heads);

/*
 * Synchronises `stream`, then reads and clears this device's status word.
 * TPMLP_OK, TPMLP_ERR_TIMEOUT (a device-side wait gave up), TPMLP_ERR_DEVICE (another
 * recorded device error) or TPMLP_ERR_CUDA.
 */
tpmlp_status tpmlp_device_status(void* stream);

/*
 * Test hook for the bounded waits: launches one warp that waits on a barrier
 * nothing completes, with a limit of timeout_us microseconds (1 .. 1000000).
 * The wait gives up, records TPMLP_ERR_TIMEOUT in the status word and returns.
 */
tpmlp_status tpmlp_debug_wait_timeout(uint32_t timeout_us, void* stream);

/*
 * Optional side stream for the fused backwards (tpmlp_mlp_bwd, tpmlp_mlp_bwd_partial,
 * tpmlp_swiglu_mlp_bwd), for bf16 tensors.  With a stream and two events of the caller's
 * registered here:
 *   - tpmlp_mlp_bwd and tpmlp_mlp_bwd_partial run their two pairs of independent GEMMs side
 *     by side, each GEMM on a share of the SMs, where that is clearly faster than one after
 *     the other (GEMMs of one or two waves of tiles, e.g. s=512 b=4 h=1024 ffn=4096 p=4):
 *     dH_i on `stream` beside dB_i (then db2) on the side stream, then dA_i (after db1) on
 *     `stream` beside dX on the side stream;
 *   - otherwise (and in tpmlp_swiglu_mlp_bwd), where dB_i or dA_i (the packed dW_i) runs
 *     its last partial wave as a second launch (split-K CTA pairs, four CTAs per tile) that
 *     leaves at least half the SMs idle (e.g. s=2048 b=4 h=5120 ffn=20480 p=4: 4 tiles on 16
 *     SMs), the bias-gradient column sums (db1 = 1^T dH, db2 = 1^T dZ), which need no tensor
 *     cores, run on the side stream beside that last wave: db2 beside dB_i's and db1 beside
 *     dA_i's, or both beside the one there is; `stream` waits for them before its next GEMM;
 *   - otherwise the column sums run on the side stream beside the first of the dA and dX
 *     GEMMs whose grid leaves enough SMs idle for all of them; where no GEMM does, they run
 *     in line.
 * The side stream waits for an event recorded on `stream` before its first kernel (for dX,
 * after dH; for sums beside a last wave, between that GEMM's two launches), and `stream`
 * waits for an event recorded on the side stream after its last, so everything is
 * complete, in order, when the work enqueued on `stream` is.  With nothing
 * registered everything runs in line on `stream`.  dH, dB, dA, db1 and db2 have the same bits
 * either way; dX, where it runs side by side, may differ in the last place of a few values
 * (its fp32 partial sums added in another order).
 *   The registration is per host thread and bound to the device current at this call;
 *   the stream must belong to that device.  The library never creates, destroys or
 *   synchronises these objects: the caller keeps them alive while registered (events
 *   created with cudaEventDisableTiming suffice).  All three NULL clears it.
 *   TPMLP_ERR_NULL if only some are NULL; TPMLP_ERR_CUDA if no device can be queried.
 */
tpmlp_status tpmlp_set_side_stream(void* side_stream, void* fork_event, void* join_event);

/*
 * Tiling of the bf16 GEMMs, process wide.  0 = automatic (default): 256x256 tiles
 * on CTA pairs when there are enough of them to fill the GPU, else single-CTA
 * tiles (128x256, or 128x128 when 128x256 tiles would leave more than half of the
 * SMs idle); CTA-pair tiles store their outputs directly from registers, or, when
 * a tile's K loop is short (at most 40 blocks of 64), through shared memory with
 * TMA stores.  1 = single-CTA tiles only; 2 = CTA-pair tiles only (epilogue chosen
 * as in 0); 3 = CTA-pair tiles, direct stores; 4 = CTA-pair tiles, TMA stores (the
 * SwiGLU epilogues, and the later launches of a split contraction that add to their
 * output, always store directly).  Every TMA load lands in the shared memory of the
 * CTA that issues it (no cluster multicast).  Results agree within rounding in every
 * mode; the control exists for tuning and tests.  TPMLP_ERR_SHAPE for other values.
 */
tpmlp_status tpmlp_set_gemm_mode(int mode);
int tpmlp_get_gemm_mode(void);

/*
 * Raster order of the output tiles, process wide: tiles are visited in groups
 * of group_m consecutive M-blocks (all N-blocks of a group before the next
 * group), so that CTAs running at the same time share operand panels in L2.
 * Default 16; 1..1024, else TPMLP_ERR_SHAPE.  Affects speed only.
 */
tpmlp_status tpmlp_set_gemm_raster(int group_m);
int tpmlp_get_gemm_raster(void);

/*
 * Longest contraction, in blocks of 64, that one GEMM launch accumulates in the tensor
 * cores, process wide.  The tensor cores' fp32 accumulation error grows about linearly
 * with the number of MMA steps, so GEMMs with an fp32 output and a longer K (the weight
 * gradients dA, dB and the projections' dW over more tokens than 64 * k_blocks) run as
 * one launch per K chunk, each later one adding its partial product to the fp32 output
 * (deterministic order).  Default 4096 (262144 tokens); 0 restores it; 1..2^24, else
 * TPMLP_ERR_SHAPE.  bf16-output GEMMs are never split.
 */
tpmlp_status tpmlp_set_k_chunk(int k_blocks);
int tpmlp_get_k_chunk(void);

/* Human-readable name of a status code. */
const char* tpmlp_status_string(tpmlp_status st);

/* Thread-local description of the last failure in this thread ("" if none). */
const char* tpmlp_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int tpmlp_version(void);

/* Number of kernels this library has launched in this process, on any thread, stream
 * or device, since it was loaded: one per launch the runtime accepted, counted on the
 * host when the launch is enqueued (not when it runs).  A call rejected by argument
 * validation launches and counts nothing.  The difference of two readings around a
 * region is how many of this library's kernels the region enqueued. */
uint64_t tpmlp_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* TPMLP_H */

/*
 * ORACLE - test infrastructure only.
 *
 * A plain, slow, fp64 CPU statement of what the tensor-parallel Transformer MLP
 * block computes.  Only the tests, the smoke check and the benchmark's CPU
 * baseline may load this library; the product path never does.  It shares no
 * code, header or table with the CUDA library.
 *
 * Sources (web pages on Megatron tensor parallelism):
 *   [CP]  "列并行" (column parallelism) article, aiqz.cc
 *   [M2]  "Megatron 专家面试题 Level 2: Tensor Parallel 与 Sequence Parallel"
 *         (M025-M040), blog.cptz.space
 *   [TI]  "腾讯混元 AI Infra 一面: 张量并行/数据并行/流水线并行的连续追问",
 *         mj.mianlingai.com, answer section (参考解析)
 *   [DP]  "分布式并行训练全景: TP/PP/DP 与 DeepSpeed ZeRO 1/2/3",
 *         talentme.airsota.com, 考点 2 and 第三章
 *
 * What it computes.  The pages state that the sharded block reaches exactly
 * the unsharded result ([CP] 数学基础: the column split equation holds with
 * strict equality; [CP] MLP 应用: GeLU is split invariant and the block is
 * GeLU(X W1) W2 with one sum at the end; [DP] 考点 2: Z = Z_1 + Z_2).  So the
 * oracle is the unsharded definition, evaluated in fp64:
 *
 *   H = X A + 1 b1^T          X [M,h], A [h,f]  (Y = XW with W [in,out], [M2] M025)
 *   Y = GeLU(H)               GeLU(z) = z Phi(z)  ([CP] MLP 应用, GeLU 定义)
 *   Z = Y B + 1 b2^T          B [f,h]
 *
 * and its gradients from dZ (chain rule; [M2] M025 and M026 name the local
 * weight gradients and the summed input gradient):
 *
 *   dB = Y^T dZ,  db2 = 1^T dZ,  dY = dZ B^T,  dH = dY * GeLU'(H),
 *   dA = X^T dH,  db1 = 1^T dH,  dX = dH A^T,
 *   GeLU'(z) = Phi(z) + z phi(z).
 *
 * Rows are tokens: token (s_idx, b_idx) of an [s,b,h] tensor is row
 * m = s_idx*b + b_idx.  All matrices are dense row-major.
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 * The layout helpers at the end (column shard, per-head QKV interleave) are
 * integer index maps and are pinned by brute-force checks there too.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_ACT_NONE 0
#define ORACLE_ACT_GELU 1
#define ORACLE_ACT_RELU 2 /* only to mirror the ReLU stand-in of the [DP] NumPy demo */

/* Phi(z), the standard normal CDF, written through erfc so that it keeps its
 * relative accuracy for negative z: Phi(z) = erfc(-z / sqrt 2) / 2. */
static double std_normal_cdf(double z) { return 0.5 * erfc(-z * 0.70710678118654752440084436210485); }

/* phi(z) = exp(-z^2/2) / sqrt(2 pi) */
static double std_normal_pdf(double z) { return 0.39894228040143267793994605993438 * exp(-0.5 * z * z); }

/* [CP] MLP 应用: GeLU(z) = z * Phi(z) */
double oracle_gelu(double z) { return z * std_normal_cdf(z); }

/* d/dz [z Phi(z)] = Phi(z) + z phi(z) */
double oracle_gelu_grad(double z) { return std_normal_cdf(z) + z * std_normal_pdf(z); }

static double act_fwd(int act, double z) {
    switch (act) {
    case ORACLE_ACT_GELU: return oracle_gelu(z);
    case ORACLE_ACT_RELU: return z > 0.0 ? z : 0.0;
    default: return z;
    }
}

static double act_grad(int act, double z) {
    switch (act) {
    case ORACLE_ACT_GELU: return oracle_gelu_grad(z);
    case ORACLE_ACT_RELU: return z > 0.0 ? 1.0 : 0.0;
    default: return 1.0;
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* C[M,N] = A[M,K] B[K,N]; plain i-k-j loops, rows in parallel. */
static void matmul_nn(int64_t M, int64_t K, int64_t N, const double* A, const double* B, double* C) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        double* c = C + i * N;
        for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = A[i * K + k];
            const double* b = B + k * N;
            for (int64_t j = 0; j < N; ++j) c[j] += a * b[j];
        }
    }
}

/* C[M,N] = A[M,K] B[N,K]^T */
static void matmul_nt(int64_t M, int64_t K, int64_t N, const double* A, const double* B, double* C) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        const double* a = A + i * K;
        for (int64_t j = 0; j < N; ++j) {
            const double* b = B + j * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += a[k] * b[k];
            C[i * N + j] = acc;
        }
    }
}

/* C[M,N] = A[K,M]^T B[K,N]  (sum over the shared leading index) */
static void matmul_tn(int64_t M, int64_t K, int64_t N, const double* A, const double* B, double* C) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        double* c = C + i * N;
        for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = A[k * M + i];
            const double* b = B + k * N;
            for (int64_t j = 0; j < N; ++j) c[j] += a * b[j];
        }
    }
}

/*
 * Forward of the unsharded block.  H, Y: [M,f]; Z: [M,h].  b1 [f] and b2 [h]
 * may be NULL (no bias).  b2 is added once, to the full sum.
 */
void oracle_mlp_fwd(int64_t M, int64_t h, int64_t f, int act,
                    const double* X, const double* A, const double* b1,
                    const double* B, const double* b2,
                    double* H, double* Y, double* Z) {
    matmul_nn(M, h, f, X, A, H); /* H = X A */
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < f; ++j) {
            double v = H[m * f + j] + (b1 ? b1[j] : 0.0);
            H[m * f + j] = v;
            Y[m * f + j] = act_fwd(act, v);
        }
    matmul_nn(M, f, h, Y, B, Z); /* Z = Y B */
    if (b2) {
#pragma omp parallel for schedule(static)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < h; ++n) Z[m * h + n] += b2[n];
    }
}

/*
 * Backward of the unsharded block from dZ [M,h], given the forward's H and Y.
 * Outputs dX [M,h], dA [h,f], dB [f,h], db1 [f], db2 [h]; db1/db2 may be NULL.
 * dH_work is caller scratch of [M,f] doubles (it holds dY, then dH).
 */
void oracle_mlp_bwd(int64_t M, int64_t h, int64_t f, int act,
                    const double* X, const double* A, const double* B,
                    const double* H, const double* Y, const double* dZ,
                    double* dX, double* dA, double* dB, double* db1, double* db2,
                    double* dH_work) {
    matmul_tn(f, M, h, Y, dZ, dB);       /* dB = Y^T dZ        [f,h] */
    matmul_nt(M, h, f, dZ, B, dH_work);  /* dY = dZ B^T        [M,f] */
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < f; ++j) dH_work[m * f + j] *= act_grad(act, H[m * f + j]);
    matmul_tn(h, M, f, X, dH_work, dA);  /* dA = X^T dH        [h,f] */
    matmul_nt(M, f, h, dH_work, A, dX);  /* dX = dH A^T        [M,h] */
    if (db1) {
        for (int64_t j = 0; j < f; ++j) db1[j] = 0.0;
        for (int64_t m = 0; m < M; ++m)
            for (int64_t j = 0; j < f; ++j) db1[j] += dH_work[m * f + j];
    }
    if (db2) {
        for (int64_t n = 0; n < h; ++n) db2[n] = 0.0;
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < h; ++n) db2[n] += dZ[m * h + n];
    }
}

/*
 * Sampled backward, for sizes where the full products are too slow.  For each
 * listed token m (rows[r]) it returns dX[m,:] as dX_rows[r,:], element by
 * element from the definitions above:
 *   H[m,j]  = X[m,:] . A[:,j] + b1[j]
 *   dH[m,j] = (dZ[m,:] . B[j,:]) * act'(H[m,j])
 *   dX[m,n] = sum_j dH[m,j] A[n,j]
 */
void oracle_bwd_dX_rows(int64_t M, int64_t h, int64_t f, int act,
                        const double* X, const double* A, const double* b1,
                        const double* B, const double* dZ,
                        int64_t n_rows, const int64_t* rows, double* dX_rows) {
    (void)M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t m = rows[r];
        double* out = dX_rows + r * h;
        for (int64_t n = 0; n < h; ++n) out[n] = 0.0;
        for (int64_t j = 0; j < f; ++j) {
            double hv = b1 ? b1[j] : 0.0;
            for (int64_t k = 0; k < h; ++k) hv += X[m * h + k] * A[k * f + j];
            double dy = 0.0;
            for (int64_t n = 0; n < h; ++n) dy += dZ[m * h + n] * B[j * h + n];
            const double dh = dy * act_grad(act, hv);
            for (int64_t n = 0; n < h; ++n) out[n] += dh * A[n * f + j];
        }
    }
}

/*
 * Sampled backward over FFN columns.  For each listed FFN index j (cols[c]):
 *   dA_cols[:, c] = dA[:, j] = sum_m X[m,:] dH[m,j]        ([h, n_cols] row-major)
 *   dB_rows[c, :] = dB[j, :] = sum_m Y[m,j] dZ[m,:]        ([n_cols, h])
 *   db1_cols[c]   = db1[j]   = sum_m dH[m,j]               (may be NULL)
 * with H, Y, dH of column j formed from the definitions above.
 */
void oracle_bwd_ffn_cols(int64_t M, int64_t h, int64_t f, int act,
                         const double* X, const double* A, const double* b1,
                         const double* B, const double* dZ,
                         int64_t n_cols, const int64_t* cols,
                         double* dA_cols, double* dB_rows, double* db1_cols) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t c = 0; c < n_cols; ++c) {
        const int64_t j = cols[c];
        double sum_dh = 0.0;
        for (int64_t n = 0; n < h; ++n) { dA_cols[n * n_cols + c] = 0.0; dB_rows[c * h + n] = 0.0; }
        for (int64_t m = 0; m < M; ++m) {
            double hv = b1 ? b1[j] : 0.0;
            for (int64_t k = 0; k < h; ++k) hv += X[m * h + k] * A[k * f + j];
            double dy = 0.0;
            for (int64_t n = 0; n < h; ++n) dy += dZ[m * h + n] * B[j * h + n];
            const double dh = dy * act_grad(act, hv);
            const double y = act_fwd(act, hv);
            sum_dh += dh;
            for (int64_t k = 0; k < h; ++k) dA_cols[k * n_cols + c] += X[m * h + k] * dh;
            for (int64_t n = 0; n < h; ++n) dB_rows[c * h + n] += y * dZ[m * h + n];
        }
        if (db1_cols) db1_cols[c] = sum_dh;
    }
}

/* db2 = 1^T dZ (the row-parallel bias gradient: b2 is added once to the summed
 * output, so its gradient is the plain column sum of dZ). */
void oracle_bwd_db2(int64_t M, int64_t h, const double* dZ, double* db2) {
    for (int64_t n = 0; n < h; ++n) db2[n] = 0.0;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < h; ++n) db2[n] += dZ[m * h + n];
}

/*
 * A single parallel linear layer, the building block of the attention
 * projections ([M2] M025 and M026: Y = X W with W [in, out]; dW = X^T dY is
 * local; dX = dY W^T; [TI]: QKV is column parallel by heads, the output
 * projection row parallel).
 *   Y = X W + 1 b^T                  X [M,K], W [K,N], b [N] (may be NULL)
 *   dX = dY W^T,  dW = X^T dY,  db = 1^T dY   (db may be NULL)
 */
void oracle_linear_fwd(int64_t M, int64_t K, int64_t N, const double* X, const double* W, const double* b,
                       double* Y) {
    matmul_nn(M, K, N, X, W, Y);
    if (b) {
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n) Y[m * N + n] += b[n];
    }
}

void oracle_linear_bwd(int64_t M, int64_t K, int64_t N, const double* X, const double* W, const double* dY,
                       double* dX, double* dW, double* db) {
    matmul_nt(M, N, K, dY, W, dX);  /* dX = dY W^T  [M,K] */
    matmul_tn(K, M, N, X, dY, dW);  /* dW = X^T dY  [K,N] */
    if (db) {
        for (int64_t n = 0; n < N; ++n) db[n] = 0.0;
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n) db[n] += dY[m * N + n];
    }
}

/*
 * SwiGLU variant of the block ([M2] M027: a gated activation such as SwiGLU
 * works on local pairs of the FFN shard, so the column + row split still needs
 * only the final sum; M031 notes its two branches as a divisibility constraint).
 * The gate G and up U projections are both column parallel:
 *   Hg = X G + 1 bg^T,  Hu = X U + 1 bu^T,  Y = silu(Hg) * Hu,  Z = Y B + 1 b2^T,
 *   silu(x) = x sigma(x),  sigma(x) = 1 / (1 + exp(-x)).
 * Backward from dZ:
 *   dB = Y^T dZ, db2 = 1^T dZ, dY = dZ B^T,
 *   dHg = dY * Hu * silu'(Hg),  silu'(x) = sigma(x) (1 + x (1 - sigma(x))),
 *   dHu = dY * silu(Hg),
 *   dG = X^T dHg, dU = X^T dHu, dbg = 1^T dHg, dbu = 1^T dHu, dX = dHg G^T + dHu U^T.
 * G, U [h,f]; bg, bu [f] (may be NULL); Hg, Hu, Y [M,f].
 */
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
double oracle_silu(double x) { return x * sigmoid(x); }
double oracle_silu_grad(double x) { const double s = sigmoid(x); return s * (1.0 + x * (1.0 - s)); }

void oracle_swiglu_fwd(int64_t M, int64_t h, int64_t f,
                       const double* X, const double* G, const double* U, const double* bg, const double* bu,
                       const double* B, const double* b2,
                       double* Hg, double* Hu, double* Y, double* Z) {
    matmul_nn(M, h, f, X, G, Hg);
    matmul_nn(M, h, f, X, U, Hu);
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < f; ++j) {
            const double g = Hg[m * f + j] + (bg ? bg[j] : 0.0);
            const double u = Hu[m * f + j] + (bu ? bu[j] : 0.0);
            Hg[m * f + j] = g;
            Hu[m * f + j] = u;
            Y[m * f + j] = oracle_silu(g) * u;
        }
    matmul_nn(M, f, h, Y, B, Z);
    if (b2) {
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < h; ++n) Z[m * h + n] = Z[m * h + n] + b2[n];
    }
}

/* work: 3 * M * f + M * h doubles of caller scratch (dY, dHg, dHu, dHu U^T). db* may be NULL. */
void oracle_swiglu_bwd(int64_t M, int64_t h, int64_t f,
                       const double* X, const double* G, const double* U, const double* B,
                       const double* Hg, const double* Hu, const double* Y, const double* dZ,
                       double* dX, double* dG, double* dU, double* dB, double* dbg, double* dbu, double* db2,
                       double* work) {
    double* dY = work;
    double* dHg = work + M * f;
    double* dHu = work + 2 * M * f;
    matmul_tn(f, M, h, Y, dZ, dB);       /* dB = Y^T dZ */
    matmul_nt(M, h, f, dZ, B, dY);       /* dY = dZ B^T */
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < f; ++j) {
            const double g = Hg[m * f + j], u = Hu[m * f + j], dy = dY[m * f + j];
            dHg[m * f + j] = dy * u * oracle_silu_grad(g);
            dHu[m * f + j] = dy * oracle_silu(g);
        }
    matmul_tn(h, M, f, X, dHg, dG);      /* dG = X^T dHg */
    matmul_tn(h, M, f, X, dHu, dU);      /* dU = X^T dHu */
    matmul_nt(M, f, h, dHg, G, dX);      /* dX = dHg G^T ... */
    double* tmp = work + 3 * M * f;      /* dHu U^T */
    matmul_nt(M, f, h, dHu, U, tmp);
    for (int64_t i = 0; i < M * h; ++i) dX[i] += tmp[i];  /* ... + dHu U^T */
    if (dbg) {
        for (int64_t j = 0; j < f; ++j) { dbg[j] = 0.0; dbu[j] = 0.0; }
        for (int64_t m = 0; m < M; ++m)
            for (int64_t j = 0; j < f; ++j) { dbg[j] += dHg[m * f + j]; dbu[j] += dHu[m * f + j]; }
    }
    if (db2) {
        for (int64_t n = 0; n < h; ++n) db2[n] = 0.0;
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < h; ++n) db2[n] += dZ[m * h + n];
    }
}

/*
 * The packed SwiGLU weight layout of the CUDA path, as an index map: each shard's
 * gate and up columns interleaved in blocks of 128 features,
 *   W_sh[i][r][256 b + j] = G[r][i fs + 128 b + j]          (j < 128)
 *                         = U[r][i fs + 128 b + j - 128]    (j >= 128),  fs = f / p.
 * inverse = 1 unpacks W_sh into G and U.
 */
void oracle_swiglu_pack(int64_t elem_size, int64_t rows, int64_t f, int64_t p, int inverse,
                        void* G, void* U, void* W_sh) {
    const int64_t fs = f / p;
    unsigned char* g = (unsigned char*)G;
    unsigned char* u = (unsigned char*)U;
    unsigned char* w = (unsigned char*)W_sh;
    for (int64_t i = 0; i < p; ++i)
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t c = 0; c < 2 * fs; ++c) {
                const int64_t blk = c / 256, j = c % 256;
                unsigned char* src = (j < 128 ? g : u) + (r * f + i * fs + 128 * blk + (j % 128)) * elem_size;
                unsigned char* dst = w + ((i * rows + r) * 2 * fs + c) * elem_size;
                if (!inverse) memcpy(dst, src, (size_t)elem_size);
                else memcpy(src, dst, (size_t)elem_size);
            }
}

/* ------------------------------------------------------------------------ */
/* Layout maps (integer index work; compared bit for bit).                   */

/*
 * Column shard ([CP] 切分原理: W = [W(1) || ... || W(p)], W(i) in R^{d x h/p};
 * [M2] M025: W_i [h, 4h/t]).  dst holds the p shards back to back, each
 * row-major:  dst[i][r][c] = src[r][i*cs + c],  cs = cols / p.
 * Elements are opaque words of elem_size bytes (2 or 4).
 */
void oracle_shard_columns(int64_t elem_size, int64_t rows, int64_t cols, int64_t p,
                          const void* src, void* dst) {
    const int64_t cs = cols / p;
    const unsigned char* s = (const unsigned char*)src;
    unsigned char* d = (unsigned char*)dst;
    for (int64_t i = 0; i < p; ++i)
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t c = 0; c < cs; ++c)
                memcpy(d + ((i * rows + r) * cs + c) * elem_size,
                       s + (r * cols + i * cs + c) * elem_size, (size_t)elem_size);
}

/*
 * Per-head interleave of a packed QKV projection ([TI] answer on QKV: lay the
 * packed matrix out so that each head's Q, K and V blocks land on the same
 * card; [M2] M028: QKV is column parallel by heads).
 *
 * Source columns: [Q | K | V], each h wide, head g of Q occupying columns
 * g*d .. g*d+d-1 (d = h / n_heads).  Destination columns: head-major
 * [q_0 k_0 v_0 | q_1 k_1 v_1 | ...], so that a column split into p equal
 * blocks hands rank r the heads r*n/p .. (r+1)*n/p - 1 with all of Q, K, V.
 *   dst column (3g + t) d + e  <-  src column t h + g d + e,  t in {0,1,2}.
 */
int64_t oracle_qkv_src_col(int64_t dst_col, int64_t h, int64_t n_heads) {
    const int64_t d = h / n_heads;
    const int64_t blk = dst_col / d;  /* 3g + t */
    const int64_t e = dst_col % d;
    const int64_t g = blk / 3, t = blk % 3;
    return t * h + g * d + e;
}

/* dst[r][c] = src[r][qkv_src_col(c)]  (inverse = 0), or the transpose map. */
void oracle_qkv_interleave(int64_t elem_size, int64_t rows, int64_t h, int64_t n_heads, int inverse,
                           const void* src, void* dst) {
    const int64_t cols = 3 * h;
    const unsigned char* s = (const unsigned char*)src;
    unsigned char* d = (unsigned char*)dst;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            const int64_t sc = oracle_qkv_src_col(c, h, n_heads);
            if (!inverse)
                memcpy(d + (r * cols + c) * elem_size, s + (r * cols + sc) * elem_size, (size_t)elem_size);
            else
                memcpy(d + (r * cols + sc) * elem_size, s + (r * cols + c) * elem_size, (size_t)elem_size);
        }
}

// fp32 FMA GEMM (the fp32 path: no TF32, so results stay within fp32 rounding),
// column sums for the bias gradients, bit-exact layout copies and the
// bounded-wait test hook.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace tpmlp {
namespace {

// ------------------------------------------------------------------ fp32 GEMM
struct SimtArgs {
    int M, N, K, n_shards, sum_shards, a_batched, b_batched;
    const float* a; long long a_ld, a_ss; int a_mn;
    const float* b; long long b_ld, b_ss; int b_mn;
    int epi, act;
    float* out; long long out_ld, out_ss;
    float* out2; long long out2_ld, out2_ss;
    const float* bias; long long bias_ss;
    const float* aux; long long aux_ld, aux_ss;
};

constexpr int ST = 64, SK = 16;

__device__ __forceinline__ float gelu_f(float x) { return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f)); }
__device__ __forceinline__ float gelu_grad_f(float x) {
    return 0.5f * (1.0f + erff(x * 0.70710678118654752f)) + x * 0.39894228040143268f * expf(-0.5f * x * x);
}

__global__ void __launch_bounds__(256) simt_gemm_kernel(const SimtArgs p) {
    __shared__ float sa[SK][ST + 1];
    __shared__ float sb[SK][ST + 1];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int m0 = blockIdx.x * ST, n0 = blockIdx.y * ST;  // M-blocks on x (no 65535 limit)
    const int shard = p.sum_shards ? 0 : blockIdx.z;
    float acc[4][4] = {};
    const int n_k_shards = p.sum_shards ? p.n_shards : 1;
    for (int ksh = 0; ksh < n_k_shards; ++ksh) {
        const int sa_idx = p.sum_shards ? ksh : (p.a_batched ? shard : 0);
        const int sb_idx = p.sum_shards ? ksh : (p.b_batched ? shard : 0);
        const float* A = p.a + sa_idx * p.a_ss;
        const float* B = p.b + sb_idx * p.b_ss;
        for (int k0 = 0; k0 < p.K; k0 += SK) {
            for (int i = threadIdx.x; i < SK * ST; i += 256) {
                const int kk = i / ST, mm = i % ST;
                const int gm = m0 + mm, gk = k0 + kk;
                float va = 0.f;
                if (gm < p.M && gk < p.K) va = p.a_mn ? A[(long long)gk * p.a_ld + gm] : A[(long long)gm * p.a_ld + gk];
                sa[kk][mm] = va;
                const int gn = n0 + mm;
                float vb = 0.f;
                if (gn < p.N && gk < p.K) vb = p.b_mn ? B[(long long)gk * p.b_ld + gn] : B[(long long)gn * p.b_ld + gk];
                sb[kk][mm] = vb;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < SK; ++kk) {
                float ra[4], rb[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) ra[i] = sa[kk][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) rb[j] = sb[kk][tx * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ra[i], rb[j], acc[i][j]);
            }
            __syncthreads();
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int gm = m0 + ty * 4 + i;
        if (gm >= p.M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int gn = n0 + tx * 4 + j;
            if (gn >= p.N) continue;
            float v = acc[i][j];
            if (p.epi == EPI_BIAS_ACT) {
                if (p.bias) v += p.bias[shard * p.bias_ss + gn];
                if (p.out2) p.out2[shard * p.out2_ss + (long long)gm * p.out2_ld + gn] = v;
                if (p.act == TPMLP_ACT_GELU_ERF) v = gelu_f(v);
            } else if (p.epi == EPI_DGELU) {
                v *= gelu_grad_f(p.aux[shard * p.aux_ss + (long long)gm * p.aux_ld + gn]);
            }
            p.out[shard * p.out_ss + (long long)gm * p.out_ld + gn] = v;
        }
    }
}

// ------------------------------------------------------------------ column sums
// out[s][n] = sum_m in[s][m][n], rows summed in a fixed order (deterministic).
template <bool IN_F32, bool OUT_F32>
__global__ void __launch_bounds__(256) colsum_kernel(const void* in, long long M, long long N, void* out) {
    __shared__ float part[8][64];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const long long s = blockIdx.y;
    const long long c = (long long)blockIdx.x * 64 + tx * 2;
    float a0 = 0.f, a1 = 0.f;
    if (c < N) {
        for (long long m = ty; m < M; m += 8) {
            const long long off = (s * M + m) * N + c;
            if (IN_F32) {
                const float2 v = *reinterpret_cast<const float2*>(static_cast<const float*>(in) + off);
                a0 += v.x;
                a1 += v.y;
            } else {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(in) + off);
                a0 += __uint_as_float(w << 16);
                a1 += __uint_as_float(w & 0xFFFF0000u);
            }
        }
    }
    part[ty][tx * 2] = a0;
    part[ty][tx * 2 + 1] = a1;
    __syncthreads();
    if (ty == 0 && c < N) {
        float r0 = 0.f, r1 = 0.f;
        for (int i = 0; i < 8; ++i) {
            r0 += part[i][tx * 2];
            r1 += part[i][tx * 2 + 1];
        }
        if (OUT_F32) {
            float* o = static_cast<float*>(out) + s * N + c;
            o[0] = r0;
            o[1] = r1;
        } else {
            __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out) + s * N + c;
            o[0] = __float2bfloat16_rn(r0);
            o[1] = __float2bfloat16_rn(r1);
        }
    }
}

// Column sums of a bf16 [shards][M][N] tensor: a cluster of 8 CTAs shares one
// 256-column strip; each CTA has 16 warps, warp w of CTA g summing rows
// 16 g + w + 128 i, eight 16-byte loads in flight per thread (enough bytes in flight
// for HBM even with a single shard, i.e. about one CTA per SM).  The partial sums are
// added in shared memory and then across the cluster's shared memory in a fixed
// order, so the result is deterministic and needs no global scratch.  (N is a
// multiple of 8.)
constexpr int CS_CLUSTER = 8;
constexpr int CS_WARPS = 16;
template <bool OUT_F32>
__global__ void __cluster_dims__(1, CS_CLUSTER, 1) __launch_bounds__(CS_WARPS * 32)
    colsum_bf16_cluster_kernel(const __nv_bfloat16* __restrict__ in, long long M, long long N, void* out) {
    namespace cg = cooperative_groups;
    __shared__ float part[CS_WARPS][256];
    __shared__ float block_sum[256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long s = blockIdx.z;
    const long long c = (long long)blockIdx.x * 256 + lane * 8;
    const int grp = blockIdx.y;  // == rank in the cluster
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (c < N) {
        const __nv_bfloat16* base = in + s * M * N + c;
#pragma unroll 8
        for (long long m = (long long)grp * CS_WARPS + warp; m < M; m += CS_WARPS * CS_CLUSTER) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(base + m * N));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] += __uint_as_float(w[i] << 16);
                acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) part[warp][lane * 8 + i] = acc[i];
    __syncthreads();
    if (threadIdx.x < 256) {
        float r = 0.f;
        for (int w = 0; w < CS_WARPS; ++w) r += part[w][threadIdx.x];
        block_sum[threadIdx.x] = r;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();  // every CTA's block_sum is complete
    if (grp == 0 && threadIdx.x < 256) {
        float r = 0.f;
        for (int g = 0; g < CS_CLUSTER; ++g) r += cluster.map_shared_rank(block_sum, g)[threadIdx.x];
        const long long col = (long long)blockIdx.x * 256 + threadIdx.x;
        if (col < N) {
            if (OUT_F32) static_cast<float*>(out)[s * N + col] = r;
            else static_cast<__nv_bfloat16*>(out)[s * N + col] = __float2bfloat16_rn(r);
        }
    }
    cluster.sync();  // peers stay resident until CTA 0 has read their shared memory
}

// The same column sums without a cluster: one CTA per 256-column strip and shard does the work
// of the 8-CTA cluster above in the same order (accumulator set g holds what CTA g of the
// cluster sums: warp w takes rows 16 g + w + 128 i in increasing order; then each set is added
// over the 16 warps, and the sets over g), so the results are bit-identical to that kernel's,
// and any free SM can run it, e.g. beside a GEMM whose last wave leaves SMs idle.
template <bool OUT_F32>
__global__ void __launch_bounds__(CS_WARPS * 32)
    colsum_bf16_strip_kernel(const __nv_bfloat16* __restrict__ in, long long M, long long N, void* out) {
    __shared__ float part[CS_WARPS][256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long s = blockIdx.z;
    const long long c = (long long)blockIdx.x * 256 + lane * 8;
    const __nv_bfloat16* base = in + s * M * N + c;
    float r = 0.f;
    // one accumulator set at a time (eight registers, as in the cluster kernel), so that
    // several CTAs fit on an SM and keep enough loads in flight
#pragma unroll 1
    for (int g = 0; g < CS_CLUSTER; ++g) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (c < N) {
#pragma unroll 8
            for (long long m = (long long)g * CS_WARPS + warp; m < M; m += CS_WARPS * CS_CLUSTER) {
                const uint4 u = __ldg(reinterpret_cast<const uint4*>(base + m * N));
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] += __uint_as_float(w[i] << 16);
                    acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) part[warp][lane * 8 + k] = acc[k];
        __syncthreads();
        if (threadIdx.x < 256) {
            float bs = 0.f;
            for (int w = 0; w < CS_WARPS; ++w) bs += part[w][threadIdx.x];
            r += bs;
        }
        __syncthreads();
    }
    const long long col = (long long)blockIdx.x * 256 + threadIdx.x;
    if (threadIdx.x < 256 && col < N) {
        if (OUT_F32) static_cast<float*>(out)[s * N + col] = r;
        else static_cast<__nv_bfloat16*>(out)[s * N + col] = __float2bfloat16_rn(r);
    }
}

// ------------------------------------------------------------------ layouts
// Column shard: dst[i][r][c] = src[r][i*cs + c] in 16-byte units (rows of cs*esize bytes).
// Each CTA takes whole rows of the unsharded layout in turn: it reads a row front to back and
// writes its p pieces, each a contiguous run of the sharded layout, with no division per unit;
// four independent units per thread and step keep enough bytes in flight.
__global__ void shard_columns_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long rows,
                                     int units_per_row /*cols*esize/16*/, int units_per_shard_row, int p,
                                     int inverse) {
    for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
        const long long row_base = r * units_per_row;
        for (int i = 0; i < p; ++i) {
            const long long a = row_base + static_cast<long long>(i) * units_per_shard_row;  // unsharded
            const long long b = (static_cast<long long>(i) * rows + r) * units_per_shard_row;  // sharded
            const uint4* from = inverse ? src + b : src + a;
            uint4* to = inverse ? dst + a : dst + b;
            int c = static_cast<int>(threadIdx.x);
            for (; c + 3 * static_cast<int>(blockDim.x) < units_per_shard_row; c += 4 * static_cast<int>(blockDim.x)) {
                const uint4 v0 = from[c], v1 = from[c + blockDim.x], v2 = from[c + 2 * blockDim.x],
                            v3 = from[c + 3 * blockDim.x];
                to[c] = v0;
                to[c + blockDim.x] = v1;
                to[c + 2 * blockDim.x] = v2;
                to[c + 3 * blockDim.x] = v3;
            }
            for (; c < units_per_shard_row; c += blockDim.x) to[c] = from[c];
        }
    }
}

// QKV interleave in units of T (16 bytes when a head's width allows): each CTA takes whole
// rows in turn; unit c of a row's head-major output is unit qkv_src_col(c) of the packed
// [Q | K | V] input (or the reverse), with 32-bit index arithmetic.
template <typename T>
__global__ void qkv_kernel(const T* __restrict__ src, T* __restrict__ dst, long long rows, int cols_units,
                           int h_units, int d_units, int inverse) {
    for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
        const T* s = src + r * cols_units;
        T* d = dst + r * cols_units;
        for (int c = static_cast<int>(threadIdx.x); c < cols_units; c += static_cast<int>(blockDim.x)) {
            const int blk = c / d_units, e = c - blk * d_units;
            const int g = blk / 3, t = blk - g * 3;
            const int sc = t * h_units + g * d_units + e;
            if (!inverse) d[c] = s[sc];
            else d[sc] = s[c];
        }
    }
}

// SwiGLU packed layout in 16-byte units (u elements each; 128 is a multiple of u):
// packed column c = 256 b + j of shard i  <->  (j < 128 ? G : U) column i fs + 128 b + j % 128.
__global__ void swiglu_pack_kernel(uint4* __restrict__ G, uint4* __restrict__ U, uint4* __restrict__ W, long long rows,
                                   long long f, long long fs, int p, int u, int inverse) {
    const long long units_per_row = 2 * fs / u;
    const long long total = (long long)p * rows * units_per_row;
    for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < total;
         x += (long long)gridDim.x * blockDim.x) {
        const long long i = x / (rows * units_per_row);
        const long long rem = x - i * rows * units_per_row;
        const long long r = rem / units_per_row;
        const long long c = (rem - r * units_per_row) * u;
        const long long blk = c >> 8, j = c & 255;
        const long long src_col = i * fs + 128 * blk + (j & 127);
        uint4* src = (j < 128 ? G : U) + (r * f + src_col) / u;
        if (!inverse) W[x] = *src;
        else *src = W[x];
    }
}

// ------------------------------------------------------------------ sum finish
// The step after an All-Reduce of fp32 partial sums: out = round(S + bias), bias added once.
// Each thread takes 8 consecutive columns (bf16 out: two 16-byte loads of S, one 16-byte bias
// load, one 16-byte store) or 4 (fp32 out), in a grid-stride loop; cols is a multiple of 8
// (bf16) or 4 (fp32), so a group never crosses a row.
template <bool OUT_F32>
__global__ void __launch_bounds__(256) sum_finish_kernel(const float* __restrict__ S, const void* __restrict__ bias,
                                                         void* __restrict__ out, long long rows, long long cols) {
    constexpr int V = OUT_F32 ? 4 : 8;
    const long long groups_per_row = cols / V;
    const long long total = rows * groups_per_row;
    for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < total;
         u += (long long)gridDim.x * blockDim.x) {
        const long long r = u / groups_per_row;
        const long long c = (u - r * groups_per_row) * V;
        const float* src = S + r * cols + c;
        if constexpr (OUT_F32) {
            float4 v = *reinterpret_cast<const float4*>(src);
            if (bias != nullptr) {
                const float4 bb = *reinterpret_cast<const float4*>(static_cast<const float*>(bias) + c);
                v.x += bb.x;
                v.y += bb.y;
                v.z += bb.z;
                v.w += bb.w;
            }
            *reinterpret_cast<float4*>(static_cast<float*>(out) + r * cols + c) = v;
        } else {
            const float4 lo = *reinterpret_cast<const float4*>(src);
            const float4 hi = *reinterpret_cast<const float4*>(src + 4);
            float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
            if (bias != nullptr) {
                const uint4 bw = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(bias) + c);
                const uint32_t w[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[2 * i] += __uint_as_float(w[i] << 16);
                    v[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
                }
            }
            uint4 o;
            uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                __nv_bfloat162 pr = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                ow[i] = *reinterpret_cast<uint32_t*>(&pr);
            }
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + r * cols + c) = o;
        }
    }
}

// ------------------------------------------------------------------ bounded-wait hook
__global__ void debug_wait_kernel(uint32_t* status, unsigned long long timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on `bar`: the wait must give up on its own.
        mbar_wait_bounded(&bar, 0, status, timeout_ns, kWhereDebug, /*watch_status=*/false);
    }
}

int grid_for(long long work, int block) {
    long long g = (work + block - 1) / block;
    if (g > 152 * 16) g = 152 * 16;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

tpmlp_status check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("%s launch: %s", what, cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    count_launch();
    return TPMLP_OK;
}

}  // namespace

tpmlp_status launch_simt_gemm(const Operand& a, const Operand& b, const GemmSpec& g, const DeviceInfo& dev,
                              cudaStream_t st) {
    (void)dev;
    SimtArgs p{};
    p.M = (int)g.M; p.N = (int)g.N; p.K = (int)g.K;
    p.n_shards = (int)g.n_shards; p.sum_shards = g.sum_shards; p.a_batched = g.a_batched; p.b_batched = g.b_batched;
    p.a = static_cast<const float*>(a.ptr); p.a_ld = a.ld; p.a_ss = a.ss; p.a_mn = a.mn_major;
    p.b = static_cast<const float*>(b.ptr); p.b_ld = b.ld; p.b_ss = b.ss; p.b_mn = b.mn_major;
    p.epi = g.epi; p.act = g.act;
    p.out = static_cast<float*>(g.out); p.out_ld = g.out_ld; p.out_ss = g.out_ss;
    p.out2 = static_cast<float*>(g.out2); p.out2_ld = g.out2_ld; p.out2_ss = g.out2_ss;
    p.bias = static_cast<const float*>(g.bias); p.bias_ss = g.bias_ss;
    p.aux = static_cast<const float*>(g.aux); p.aux_ld = g.aux_ld; p.aux_ss = g.aux_ss;
    const long long nb = (g.N + ST - 1) / ST, sh = g.sum_shards ? 1 : g.n_shards;
    if (nb > 65535 || sh > 65535) {
        set_error("fp32 GEMM: N/64 and the shard count must be at most 65535");
        return TPMLP_ERR_SHAPE;
    }
    dim3 grid((unsigned)((g.M + ST - 1) / ST), (unsigned)nb, (unsigned)sh);
    simt_gemm_kernel<<<grid, 256, 0, st>>>(p);
    return check_launch("fp32 GEMM");
}

tpmlp_status launch_colsum(const void* in, bool in_f32, int64_t shards, int64_t M, int64_t N, void* out, bool out_f32,
                           cudaStream_t st) {
    if (!in_f32) {
        dim3 g((unsigned)((N + 255) / 256), CS_CLUSTER, (unsigned)shards);
        const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(in);
        if (out_f32) colsum_bf16_cluster_kernel<true><<<g, CS_WARPS * 32, 0, st>>>(src, M, N, out);
        else colsum_bf16_cluster_kernel<false><<<g, CS_WARPS * 32, 0, st>>>(src, M, N, out);
        return check_launch("column sum");
    }
    dim3 grid((unsigned)((N + 63) / 64), (unsigned)shards);
    if (in_f32 && out_f32) colsum_kernel<true, true><<<grid, 256, 0, st>>>(in, M, N, out);
    else if (in_f32) colsum_kernel<true, false><<<grid, 256, 0, st>>>(in, M, N, out);
    else if (out_f32) colsum_kernel<false, true><<<grid, 256, 0, st>>>(in, M, N, out);
    else colsum_kernel<false, false><<<grid, 256, 0, st>>>(in, M, N, out);
    return check_launch("column sum");
}

// bf16 column sums without clusters, bit-identical to launch_colsum's: schedulable on any
// free SM, e.g. beside a GEMM that leaves SMs idle.
tpmlp_status launch_colsum_any_sm(const void* in, int64_t shards, int64_t M, int64_t N, void* out, bool out_f32,
                                  cudaStream_t st) {
    dim3 g((unsigned)((N + 255) / 256), 1, (unsigned)shards);
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(in);
    if (out_f32) colsum_bf16_strip_kernel<true><<<g, CS_WARPS * 32, 0, st>>>(src, M, N, out);
    else colsum_bf16_strip_kernel<false><<<g, CS_WARPS * 32, 0, st>>>(src, M, N, out);
    return check_launch("column sum");
}

tpmlp_status launch_shard_columns(const void* src, void* dst, int64_t rows, int64_t cols, int p, int esize,
                                  bool inverse, cudaStream_t st) {
    const long long upr = cols * esize / 16, upsr = upr / p;
    if (upr > INT32_MAX) {
        set_error("column shard: a row of more than 2^31 16-byte units");
        return TPMLP_ERR_SHAPE;
    }
    // one row per CTA at a time; enough CTAs for every SM several times over
    const long long grid = rows < 152LL * 16 ? rows : 152LL * 16;
    shard_columns_kernel<<<static_cast<unsigned>(grid > 0 ? grid : 1), 256, 0, st>>>(
        static_cast<const uint4*>(src), static_cast<uint4*>(dst), rows, static_cast<int>(upr), static_cast<int>(upsr), p,
        inverse ? 1 : 0);
    return check_launch("column shard");
}

tpmlp_status launch_qkv_interleave(const void* src, void* dst, int64_t rows, int64_t h, int64_t n_heads, int esize,
                                   bool inverse, cudaStream_t st) {
    const long long d = h / n_heads;
    const long long cols = 3 * h;
    if (cols > INT32_MAX) {
        set_error("QKV interleave: rows of more than 2^31 elements");
        return TPMLP_ERR_SHAPE;
    }
    const unsigned grid = static_cast<unsigned>(rows < 152LL * 16 ? (rows > 0 ? rows : 1) : 152LL * 16);  // rows per CTA in turn
    if ((d * esize) % 16 == 0) {
        const long long k = 16 / esize;  // elements per unit
        qkv_kernel<uint4><<<grid, 256, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), rows,
                                               static_cast<int>(cols / k), static_cast<int>(h / k),
                                               static_cast<int>(d / k), inverse ? 1 : 0);
    } else if (esize == 2) {
        qkv_kernel<uint16_t><<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst), rows,
                                                  static_cast<int>(cols), static_cast<int>(h), static_cast<int>(d),
                                                  inverse ? 1 : 0);
    } else {
        qkv_kernel<uint32_t><<<grid, 256, 0, st>>>(static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst), rows,
                                                  static_cast<int>(cols), static_cast<int>(h), static_cast<int>(d),
                                                  inverse ? 1 : 0);
    }
    return check_launch("QKV interleave");
}

tpmlp_status launch_swiglu_pack(void* G, void* U, void* W_sh, int64_t rows, int64_t ffn, int p, int esize,
                                bool inverse, cudaStream_t st) {
    const int u = 16 / esize;
    const long long fs = ffn / p;
    const long long total = (long long)p * rows * (2 * fs / u);
    swiglu_pack_kernel<<<grid_for(total, 256), 256, 0, st>>>(static_cast<uint4*>(G), static_cast<uint4*>(U),
                                                              static_cast<uint4*>(W_sh), rows, ffn, fs, p, u,
                                                              inverse ? 1 : 0);
    return check_launch("SwiGLU pack");
}

tpmlp_status launch_sum_finish(const float* S, const void* bias, void* out, int64_t rows, int64_t cols, bool out_f32,
                               int sm_count, cudaStream_t st) {
    const long long groups = rows * (cols / (out_f32 ? 4 : 8));
    long long blocks = (groups + 255) / 256;
    const long long cap = static_cast<long long>(sm_count > 0 ? sm_count : 1) * 8;  // 8 x 256 threads per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (out_f32) sum_finish_kernel<true><<<(unsigned)blocks, 256, 0, st>>>(S, bias, out, rows, cols);
    else sum_finish_kernel<false><<<(unsigned)blocks, 256, 0, st>>>(S, bias, out, rows, cols);
    return check_launch("sum finish");
}

tpmlp_status launch_debug_wait(uint32_t timeout_us, uint32_t* status, cudaStream_t st) {
    debug_wait_kernel<<<1, 32, 0, st>>>(status, static_cast<unsigned long long>(timeout_us) * 1000ull);
    return check_launch("debug wait");
}

}  // namespace tpmlp

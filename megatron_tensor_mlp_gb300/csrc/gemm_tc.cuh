// Persistent, warp-specialised bf16 GEMM on the 5th-generation tensor cores
// (tcgen05.mma, fp32 accumulators in tensor memory), fed by TMA, with the
// fused epilogues of the tensor-parallel MLP block.
//
//   D_s[M,N] = A_s[M,K] B_s[K,N]           (batched over shards s), or
//   D  [M,N] = sum_s A_s[M,K] B_s[K,N]     (shard sum inside the K loop)
//
// Two kernels share one structure: gemm_pair_kernel (a cluster of two CTAs,
// 256x256 tiles with tcgen05.mma.cta_group::2; the main path) and gemm_kernel
// (one CTA, 128x256 or 128x128 tiles; GEMMs too small to fill the GPU with
// pair tiles).  CTA layout (384 threads, or 256 for the pair kernel's
// direct-store variant; one CTA per SM, persistent over output tiles):
//   warp 0        TMA producer: fills a ring of (A, B) stages
//   warp 1        TMEM allocator + MMA issuer (one thread): 4 UMMAs per
//                 64-wide K block into one of two fp32 accumulators
//                 (double buffered across tiles)
//   warps 2-3     idle
//   warps 4-11    epilogue: tcgen05.ld 32 columns at a time, fused
//                 bias / GeLU / GeLU' / conversion, then either 16/32-byte
//                 global stores per row or (pair kernel, short K loops)
//                 swizzled shared-memory boxes written with TMA stores;
//                 warp w reads TMEM lanes 32*(w%4).. and column half (w-4)/4
//                 (pair kernel, direct stores: warps 4-7, both halves).
// Every wait on an mbarrier is bounded (a status word records a timeout).
// Set-up runs before griddepcontrol.wait, so it overlaps the previous launch.
//
// Shared-memory operand layouts are the canonical 128-byte-swizzled ones:
//   K-major tile  : rows of 64 K-elements (128 B), 8-row atoms of 1 KiB,
//                   stride-dimension offset 1 KiB; the K step of one UMMA
//                   (16 elements = 32 B) advances the start address.
//   MN-major tile : 64-element MN chunks (128 B) x BK K-rows, one TMA box
//                   per chunk; leading-dimension offset = chunk pitch
//                   (BK * 128 B), stride-dimension offset = 8 K-rows (1 KiB);
//                   the K step advances the start address by 16 rows (2 KiB).
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace tpmlp {
namespace tc {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;                  // single-CTA 128x256 tiles: 48 KiB stages
constexpr int A_TILE_BYTES = BM * BK * 2;  // 16 KiB
constexpr int MN_CHUNK_BYTES = BK * 128;   // one 64-wide MN chunk of an MN-major tile
constexpr int NUM_THREADS = 384;
constexpr int FIRST_EPI_WARP = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr uint32_t TMEM_COLS = 512;        // two 256-column fp32 accumulators
constexpr int BAR_BYTES = 256;

#ifndef TPMLP_MN_LBO_BYTES
#define TPMLP_MN_LBO_BYTES MN_CHUNK_BYTES
#endif
#ifndef TPMLP_MN_SBO_BYTES
#define TPMLP_MN_SBO_BYTES 1024
#endif

struct KArgs {
    int M, N, K;
    int n_shards, sum_shards, a_batched, b_batched;
    int m_blocks, n_blocks, batch, num_tiles, kb_per_shard, k_iters, group_m;
    int act, out_f32;
    int a_chunked, b_chunked;  // MN-major operand loaded with one 4-D box per stage (MN extent % 64 == 0)
    int st32;                  // out, out2 and aux rows are 32-byte aligned: 32-byte global accesses
    int accumulate;            // EPI_STORE, fp32 out: out += acc (a later K chunk of a split contraction)
    int tile_begin;            // pair and split-K kernels: this launch covers tiles [tile_begin, num_tiles)
    int rev_period;            // pair kernel: tile t walks K backwards when (t / rev_period) is odd (INT_MAX: never)
    void* out; long long out_ld, out_ss;
    void* out2; long long out2_ld, out2_ss;
    const void* bias; long long bias_ss;
    const void* aux; long long aux_ld, aux_ss;
    uint32_t* status;
    unsigned long long timeout_ns;
};

__device__ __forceinline__ void decode_tile(const KArgs& p, int t, int& mb, int& nb, int& shard) {
    const int n_total = p.batch * p.n_blocks;
    const int per_group = p.group_m * n_total;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int gm = min(p.m_blocks - first_m, p.group_m);
    const int r = t - g * per_group;
    mb = first_m + r % gm;
    const int nbg = r / gm;
    shard = nbg / p.n_blocks;
    nb = nbg - shard * p.n_blocks;
}

// ---------------------------------------------------------------------------
// GeLU(x) = x Phi(x) and GeLU'(x) = Phi(x) + x phi(x), two elements at a time.
//
// Phi comes from the complementary error function, evaluated with Hastings'
// rational approximation as tabulated by Abramowitz & Stegun, "Handbook of
// Mathematical Functions", formula 7.1.26:
//     erfc(z) ~= t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2),
//     t = 1 / (1 + p z),  z >= 0,  |error| <= 1.5e-7,
// with p = 0.3275911, a1..a5 = 0.254829592, -0.284496736, 1.421413741,
// -1.453152027, 1.061405429.  With z = |x| / sqrt(2):
//     Phi(x) = 1 - erfc(z) / 2  (x >= 0),   erfc(z) / 2  (x < 0),
// and exp(-z^2) = exp(-x^2 / 2) = sqrt(2 pi) phi(x), shared by GeLU'.
// The factor 1/2 is folded into a1..a5.  The polynomial runs on packed
// fp32x2 FMAs; the reciprocal and exp2 use the hardware approximations.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Phi(x) and exp(-x^2/2) for two elements.
__device__ __forceinline__ void normal_cdf_pair(float x0, float x1, float& cdf0, float& cdf1, float& e0, float& e1) {
    const float kInvSqrt2 = 0.70710678118654752f;
    const unsigned long long z = f2_pack(fabsf(x0) * kInvSqrt2, fabsf(x1) * kInvSqrt2);
    float s0, s1;
    f2_unpack(f2_fma(f2_pack(0.3275911f, 0.3275911f), z, f2_pack(1.0f, 1.0f)), s0, s1);
    const unsigned long long t = f2_pack(rcp_approx(s0), rcp_approx(s1));
    unsigned long long q = f2_fma(t, f2_pack(0.5307027145f, 0.5307027145f), f2_pack(-0.7265760135f, -0.7265760135f));
    q = f2_fma(t, q, f2_pack(0.7107068705f, 0.7107068705f));
    q = f2_fma(t, q, f2_pack(-0.142248368f, -0.142248368f));
    q = f2_fma(t, q, f2_pack(0.127414796f, 0.127414796f));
    q = f2_mul(t, q);  // erfc(z) / 2 without the exponential
    float w0, w1;      // -z^2 log2(e) = -x^2 / 2 log2(e)
    f2_unpack(f2_mul(f2_mul(z, z), f2_pack(-1.4426950408889634f, -1.4426950408889634f)), w0, w1);
    e0 = ex2_approx(w0);
    e1 = ex2_approx(w1);
    float h0, h1;
    f2_unpack(f2_mul(q, f2_pack(e0, e1)), h0, h1);  // erfc(z) / 2
    cdf0 = x0 >= 0.0f ? 1.0f - h0 : h0;
    cdf1 = x1 >= 0.0f ? 1.0f - h1 : h1;
}

// v[j] <- GeLU(v[j]) for j in [0, 32), as max(x, 0) - |x| h with h = erfc(|x| / sqrt(2)) / 2,
// which holds for either sign (x >= 0: x Phi(x) = x - x h; x < 0: x Phi(x) = x h = -|x| h): no
// sign select, and a single rounding where x >= 0.  1/sqrt(2) is folded into p, and
// -z^2 log2(e) is taken from x directly: about 14 operations per pair of elements besides the
// four special-function ones, against 18 through normal_cdf_pair.
__device__ __forceinline__ void gelu_inplace32(float* v) {
    const float kP = 0.3275911f * 0.70710678118654752f;
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float x0 = v[j], x1 = v[j + 1];
        const unsigned long long t =
            f2_pack(rcp_approx(fmaf(kP, fabsf(x0), 1.0f)), rcp_approx(fmaf(kP, fabsf(x1), 1.0f)));
        unsigned long long q = f2_fma(t, f2_pack(0.5307027145f, 0.5307027145f), f2_pack(-0.7265760135f, -0.7265760135f));
        q = f2_fma(t, q, f2_pack(0.7107068705f, 0.7107068705f));
        q = f2_fma(t, q, f2_pack(-0.142248368f, -0.142248368f));
        q = f2_fma(t, q, f2_pack(0.127414796f, 0.127414796f));
        q = f2_mul(t, q);  // erfc(|x| / sqrt 2) / 2 without the exponential
        const unsigned long long xx = f2_pack(x0, x1);
        float w0, w1;  // -x^2 / 2 log2(e)
        f2_unpack(f2_mul(f2_mul(xx, xx), f2_pack(-0.72134752044448170f, -0.72134752044448170f)), w0, w1);
        float h0, h1;
        f2_unpack(f2_mul(q, f2_pack(ex2_approx(w0), ex2_approx(w1))), h0, h1);
        v[j] = fmaf(-fabsf(x0), h0, fmaxf(x0, 0.0f));
        v[j + 1] = fmaf(-fabsf(x1), h1, fmaxf(x1, 0.0f));
    }
}

// v[j] <- v[j] * GeLU'(h[j]) for j in [0, 8)
__device__ __forceinline__ void dgelu_mul8(float* v, const float* h) {
    const unsigned long long inv_sqrt_2pi = f2_pack(0.39894228040143268f, 0.39894228040143268f);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        float c0, c1, e0, e1;
        normal_cdf_pair(h[j], h[j + 1], c0, c1, e0, e1);
        // GeLU' = Phi + x exp(-x^2/2) / sqrt(2 pi)
        const unsigned long long g = f2_fma(f2_mul(f2_pack(h[j], h[j + 1]), f2_pack(e0, e1)), inv_sqrt_2pi,
                                            f2_pack(c0, c1));
        f2_unpack(f2_mul(f2_pack(v[j], v[j + 1]), g), v[j], v[j + 1]);
    }
}

// sigma(x) = 1 / (1 + 2^(-x log2 e)) with the hardware approximations; silu(x) = x sigma(x),
// silu'(x) = sigma(x) (1 + x (1 - sigma(x))).
__device__ __forceinline__ float sigmoid_approx(float x) {
    return rcp_approx(1.0f + ex2_approx(-1.4426950408889634f * x));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// 32-byte global accesses (Blackwell): half as many store / load instructions per row as
// 16-byte ones, so the epilogue puts half as many requests through the SM's load/store
// data pipe, which the tensor cores' shared-memory operand reads also use.  Addresses must
// be 32-byte aligned (KArgs::st32).
__device__ __forceinline__ void st_v8(void* p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4,
                                      uint32_t a5, uint32_t a6, uint32_t a7) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0), "r"(a1), "r"(a2),
                 "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
                 : "memory");
}
__device__ __forceinline__ void ld_v8(const void* p, uint32_t (&w)[8]) {
    asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p)
                 : "memory");
}

// Store 32 values (nvalid is a multiple of 8) as bf16: with st32 in 32-byte groups of 16
// (a trailing group of 8 as one 16-byte store), else in 16-byte groups of 8.
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v, int nvalid, bool st32) {
    if (st32) {
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const float* w = v + g * 16;
            if ((g + 1) * 16 <= nvalid) {
                st_v8(dst + g * 16, pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]), pack_bf16x2(w[4], w[5]),
                      pack_bf16x2(w[6], w[7]), pack_bf16x2(w[8], w[9]), pack_bf16x2(w[10], w[11]),
                      pack_bf16x2(w[12], w[13]), pack_bf16x2(w[14], w[15]));
            } else if (g * 16 < nvalid) {
                uint4 u;
                u.x = pack_bf16x2(w[0], w[1]);
                u.y = pack_bf16x2(w[2], w[3]);
                u.z = pack_bf16x2(w[4], w[5]);
                u.w = pack_bf16x2(w[6], w[7]);
                *reinterpret_cast<uint4*>(dst + g * 16) = u;
            }
        }
        return;
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (g * 8 < nvalid) {
            uint4 u;
            u.x = pack_bf16x2(v[g * 8 + 0], v[g * 8 + 1]);
            u.y = pack_bf16x2(v[g * 8 + 2], v[g * 8 + 3]);
            u.z = pack_bf16x2(v[g * 8 + 4], v[g * 8 + 5]);
            u.w = pack_bf16x2(v[g * 8 + 6], v[g * 8 + 7]);
            *reinterpret_cast<uint4*>(dst + g * 8) = u;
        }
    }
}
// Store 32 fp32 values (nvalid is a multiple of 4): 32-byte groups of 8 with st32, else 16-byte.
__device__ __forceinline__ void store_f32x32(float* dst, const float* v, int nvalid, bool st32) {
    if (st32) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const float* w = v + g * 8;
            if ((g + 1) * 8 <= nvalid) {
                st_v8(dst + g * 8, __float_as_uint(w[0]), __float_as_uint(w[1]), __float_as_uint(w[2]),
                      __float_as_uint(w[3]), __float_as_uint(w[4]), __float_as_uint(w[5]), __float_as_uint(w[6]),
                      __float_as_uint(w[7]));
            } else if (g * 8 < nvalid) {
                *reinterpret_cast<float4*>(dst + g * 8) = make_float4(w[0], w[1], w[2], w[3]);
            }
        }
        return;
    }
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        if (g * 4 < nvalid) {
            *reinterpret_cast<float4*>(dst + g * 4) = make_float4(v[g * 4], v[g * 4 + 1], v[g * 4 + 2], v[g * 4 + 3]);
        }
    }
}
// v[j] += src[j] for the first nvalid (a multiple of 4) of 32 fp32 values of a row.
__device__ __forceinline__ void add_f32x32(const float* src, float* v, int nvalid, bool st32) {
    if (st32) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            if ((g + 1) * 8 <= nvalid) {
                uint32_t w[8];
                ld_v8(src + g * 8, w);
#pragma unroll
                for (int i = 0; i < 8; ++i) v[g * 8 + i] += __uint_as_float(w[i]);
            } else if (g * 8 < nvalid) {
                const float4 f = *reinterpret_cast<const float4*>(src + g * 8);
                v[g * 8 + 0] += f.x;
                v[g * 8 + 1] += f.y;
                v[g * 8 + 2] += f.z;
                v[g * 8 + 3] += f.w;
            }
        }
        return;
    }
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        if (g * 4 < nvalid) {
            const float4 f = *reinterpret_cast<const float4*>(src + g * 4);
            v[g * 4 + 0] += f.x;
            v[g * 4 + 1] += f.y;
            v[g * 4 + 2] += f.z;
            v[g * 4 + 3] += f.w;
        }
    }
}
// Load 32 bf16 values of a row (nvalid a multiple of 8) widened to fp32; values past nvalid
// are left untouched.
__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* src, float* f, int nvalid, bool st32) {
    if (st32) {
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            if ((g + 1) * 16 <= nvalid) {
                uint32_t w[8];
                ld_v8(src + g * 16, w);
                unpack_bf16x8(make_uint4(w[0], w[1], w[2], w[3]), f + g * 16);
                unpack_bf16x8(make_uint4(w[4], w[5], w[6], w[7]), f + g * 16 + 8);
            } else if (g * 16 < nvalid) {
                unpack_bf16x8(*reinterpret_cast<const uint4*>(src + g * 16), f + g * 16);
            }
        }
        return;
    }
#pragma unroll
    for (int g = 0; g < 4; ++g)
        if (g * 8 < nvalid) unpack_bf16x8(*reinterpret_cast<const uint4*>(src + g * 8), f + g * 8);
}

// GeLU' epilogue: 32 bf16 values of H (this thread's row, columns gn0..gn0+31) as 16 packed
// pairs, loaded ahead of the chunk that uses them (the loads of a warp touch 32 rows, so each
// costs a full memory latency; issued one chunk early they overlap the previous chunk's work,
// and the first chunk's overlap the wait for the accumulator).  Words past the row's end are
// not loaded (their values are never stored).
__device__ __forceinline__ void load_h_raw(const KArgs& p, int gm, int gn0, int shard, uint32_t (&w)[16]) {
    if (gm >= p.M) return;
    const int nvalid = p.N - gn0;
    if (nvalid <= 0) return;
    const __nv_bfloat16* hp = static_cast<const __nv_bfloat16*>(p.aux) + shard * p.aux_ss + (long long)gm * p.aux_ld + gn0;
    if (p.st32) {
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            if ((g + 1) * 16 <= nvalid) {
                uint32_t t[8];
                ld_v8(hp + g * 16, t);
#pragma unroll
                for (int i = 0; i < 8; ++i) w[g * 8 + i] = t[i];
            } else if (g * 16 < nvalid) {
                const uint4 u = *reinterpret_cast<const uint4*>(hp + g * 16);
                w[g * 8 + 0] = u.x; w[g * 8 + 1] = u.y; w[g * 8 + 2] = u.z; w[g * 8 + 3] = u.w;
            }
        }
        return;
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (g * 8 < nvalid) {
            const uint4 u = *reinterpret_cast<const uint4*>(hp + g * 8);
            w[g * 4 + 0] = u.x; w[g * 4 + 1] = u.y; w[g * 4 + 2] = u.z; w[g * 4 + 3] = u.w;
        }
    }
}

// v[j] <- v[j] * GeLU'(H[j]) for the first nvalid (a multiple of 8) of 32 values, H as loaded
// by load_h_raw.
__device__ __forceinline__ void dgelu_apply32(float* v, const uint32_t (&w)[16], int nvalid) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (g * 8 < nvalid) {
            float hv[8];
            unpack_bf16x8(make_uint4(w[g * 4 + 0], w[g * 4 + 1], w[g * 4 + 2], w[g * 4 + 3]), hv);
            dgelu_mul8(v + g * 8, hv);
        }
    }
}

template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const KArgs& p, const uint32_t (&r)[32], int gm, int gn0, int shard) {
    if (gm >= p.M) return;
    const int nvalid = p.N - gn0;
    if (nvalid <= 0) return;
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    if constexpr (EPI == EPI_BIAS_ACT) {
        if (p.bias != nullptr) {
            const __nv_bfloat16* bp = static_cast<const __nv_bfloat16*>(p.bias) + shard * p.bias_ss + gn0;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                if (g * 8 < nvalid) {
                    float bf[8];
                    unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(bp + g * 8)), bf);
#pragma unroll
                    for (int i = 0; i < 8; i += 2)
                        f2_unpack(f2_add(f2_pack(v[g * 8 + i], v[g * 8 + i + 1]), f2_pack(bf[i], bf[i + 1])),
                                  v[g * 8 + i], v[g * 8 + i + 1]);
                }
            }
        }
        if (p.out2 != nullptr) {
            __nv_bfloat16* d2 = static_cast<__nv_bfloat16*>(p.out2) + shard * p.out2_ss + (long long)gm * p.out2_ld + gn0;
            store_bf16x32(d2, v, nvalid, p.st32);
        }
        if (p.act == TPMLP_ACT_GELU_ERF) gelu_inplace32(v);
        __nv_bfloat16* d = static_cast<__nv_bfloat16*>(p.out) + shard * p.out_ss + (long long)gm * p.out_ld + gn0;
        store_bf16x32(d, v, nvalid, p.st32);
    } else if constexpr (EPI == EPI_DGELU) {
        const __nv_bfloat16* hp =
            static_cast<const __nv_bfloat16*>(p.aux) + shard * p.aux_ss + (long long)gm * p.aux_ld + gn0;
        float hv[32];
        load_bf16x32(hp, hv, nvalid, p.st32);
#pragma unroll
        for (int g = 0; g < 4; ++g)
            if (g * 8 < nvalid) dgelu_mul8(v + g * 8, hv + g * 8);
        __nv_bfloat16* d = static_cast<__nv_bfloat16*>(p.out) + shard * p.out_ss + (long long)gm * p.out_ld + gn0;
        store_bf16x32(d, v, nvalid, p.st32);
    } else {
        if (p.out_f32) {
            float* d = static_cast<float*>(p.out) + shard * p.out_ss + (long long)gm * p.out_ld + gn0;
            if (p.accumulate) add_f32x32(d, v, nvalid, p.st32);  // the earlier K chunks' sum, in fp32
            store_f32x32(d, v, nvalid, p.st32);
        } else {
            __nv_bfloat16* d = static_cast<__nv_bfloat16*>(p.out) + shard * p.out_ss + (long long)gm * p.out_ld + gn0;
            store_bf16x32(d, v, nvalid, p.st32);
        }
    }
}

// SwiGLU forward: TMEM columns [0,128) hold the gate and [128,256) the up projection of the
// same 128 features (packed layout); this thread's row, features fo..fo+31 of tile nb.
__device__ __forceinline__ void swiglu_chunk(const KArgs& p, const uint32_t (&rg)[32], const uint32_t (&ru)[32],
                                             int gm, int nb, int fo, int shard) {
    if (gm >= p.M) return;
    float g[32], u[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        g[j] = __uint_as_float(rg[j]);
        u[j] = __uint_as_float(ru[j]);
    }
    const long long pg = (long long)nb * 256 + fo;  // packed gate column (up = pg + 128)
    if (p.bias != nullptr) {
        const __nv_bfloat16* bp = static_cast<const __nv_bfloat16*>(p.bias) + shard * p.bias_ss + pg;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float bg[8], bu[8];
            unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(bp + q * 8)), bg);
            unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(bp + 128 + q * 8)), bu);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                g[q * 8 + i] += bg[i];
                u[q * 8 + i] += bu[i];
            }
        }
    }
    if (p.out2 != nullptr) {  // fp32 pre-activations: the backward multiplies by u itself
        float* d2 = static_cast<float*>(p.out2) + shard * p.out2_ss + (long long)gm * p.out2_ld + pg;
        store_f32x32(d2, g, 32, p.st32);
        store_f32x32(d2 + 128, u, 32, p.st32);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) g[j] = g[j] * sigmoid_approx(g[j]) * u[j];
    __nv_bfloat16* d = static_cast<__nv_bfloat16*>(p.out) + shard * p.out_ss + (long long)gm * p.out_ld +
                       (long long)nb * 128 + fo;
    store_bf16x32(d, g, 32, p.st32);
}

// SwiGLU dgrad: acc = dY for features f0..f0+31; packed fp32 (g, u) pre-activations from aux,
// packed bf16 (dg, du) to out:  dg = dY u silu'(g),  du = dY silu(g).
__device__ __forceinline__ void dswiglu_chunk(const KArgs& p, const uint32_t (&r)[32], int gm, int f0, int shard) {
    if (gm >= p.M || f0 >= p.N) return;
    const long long pg = (long long)(f0 >> 7) * 256 + (f0 & 127);
    const float* hp = static_cast<const float*>(p.aux) + shard * p.aux_ss + (long long)gm * p.aux_ld + pg;
    __nv_bfloat16* op = static_cast<__nv_bfloat16*>(p.out) + shard * p.out_ss + (long long)gm * p.out_ld + pg;
    float gv[32], uv[32];
    if (p.st32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t w[8];
            ld_v8(hp + q * 8, w);
#pragma unroll
            for (int i = 0; i < 8; ++i) gv[q * 8 + i] = __uint_as_float(w[i]);
            ld_v8(hp + 128 + q * 8, w);
#pragma unroll
            for (int i = 0; i < 8; ++i) uv[q * 8 + i] = __uint_as_float(w[i]);
        }
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 g4 = *reinterpret_cast<const float4*>(hp + q * 4);
            const float4 u4 = *reinterpret_cast<const float4*>(hp + 128 + q * 4);
            gv[q * 4 + 0] = g4.x; gv[q * 4 + 1] = g4.y; gv[q * 4 + 2] = g4.z; gv[q * 4 + 3] = g4.w;
            uv[q * 4 + 0] = u4.x; uv[q * 4 + 1] = u4.y; uv[q * 4 + 2] = u4.z; uv[q * 4 + 3] = u4.w;
        }
    }
    float dg[32], du[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float dy = __uint_as_float(r[j]);
        const float sg = sigmoid_approx(gv[j]);
        dg[j] = dy * uv[j] * (sg * (1.0f + gv[j] * (1.0f - sg)));
        du[j] = dy * gv[j] * sg;
    }
    store_bf16x32(op, dg, 32, p.st32);
    store_bf16x32(op + 128, du, 32, p.st32);
}

// One tile's epilogue for this warp: TMEM lane quarter q, column half `half`.
// NCH = 32-column chunks per column half of the tile: 4 for 256-wide tiles, 2 for 128-wide.
template <int EPI, int NCH = 4>
__device__ __forceinline__ void epilogue_tile(const KArgs& p, uint32_t t_row, int gm, int nb, int half, int shard) {
    if constexpr (EPI == EPI_SWIGLU) {
        static_assert(NCH == 4, "the packed SwiGLU layout needs 256-wide tiles");
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
            const int fo = half * 64 + c * 32;
            uint32_t rg[32], ru[32];
            tmem_ld_32x32b_x32(t_row + fo, rg);
            tmem_ld_32x32b_x32(t_row + 128 + fo, ru);
            tmem_ld_wait();
            swiglu_chunk(p, rg, ru, gm, nb, fo, shard);
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < NCH; ++c) {
            const int col = half * (NCH * 32) + c * 32;
            uint32_t r[32];
            tmem_ld_32x32b_x32(t_row + col, r);
            tmem_ld_wait();
            static_assert(EPI != EPI_DSWIGLU || NCH == 4, "the packed SwiGLU layout needs 256-wide tiles");
            if constexpr (EPI == EPI_DSWIGLU) dswiglu_chunk(p, r, gm, nb * BN + col, shard);
            else epilogue_chunk<EPI>(p, r, gm, nb * (NCH * 64) + col, shard);
        }
    }
}

// GeLU' epilogue of L consecutive 32-column chunks of a tile TW columns wide, starting at chunk
// jbase, for this thread's row gm; h0 holds the first chunk's H on entry.  Two chunks per loop
// trip so that the H buffers are named at compile time.
template <int L, int TW>
__device__ __forceinline__ void dgelu_chunks(const KArgs& p, uint32_t t_row, int gm, int nb, int jbase, int shard,
                                             uint32_t (&h0)[16], uint32_t (&h1)[16]) {
    static_assert(L % 2 == 0, "chunks come in pairs");
#pragma unroll 1
    for (int i = 0; i < L; i += 2) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            uint32_t(&cur)[16] = k == 0 ? h0 : h1;
            uint32_t(&nxt)[16] = k == 0 ? h1 : h0;
            const int col = (jbase + i + k) * 32;
            const int gn0 = nb * TW + col;
            if (i + k + 1 < L) load_h_raw(p, gm, gn0 + 32, shard, nxt);
            uint32_t r[32];
            tmem_ld_32x32b_x32(t_row + col, r);
            tmem_ld_wait();
            const int nvalid = p.N - gn0;
            if (gm < p.M && nvalid > 0) {
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                dgelu_apply32(v, cur, nvalid);
                __nv_bfloat16* d =
                    static_cast<__nv_bfloat16*>(p.out) + shard * p.out_ss + (long long)gm * p.out_ld + gn0;
                store_bf16x32(d, v, nvalid, p.st32);
            }
        }
    }
}

// Single-CTA tiles are BM x SBN: SBN = 256 (4-stage ring of 48 KiB), or SBN = 128 for GEMMs
// with too few 256-wide tiles to fill the SMs (7-stage ring of 32 KiB, 2 x 128 TMEM columns).
template <int SBN>
struct SingleGeom {
    static_assert(SBN == 256 || SBN == 128, "single-CTA tile width");
    static constexpr int b_bytes = SBN * BK * 2;
    static constexpr int stage_bytes = A_TILE_BYTES + b_bytes;
    static constexpr int stages = SBN == 256 ? STAGES : 7;
    static constexpr uint32_t tmem_cols = 2 * SBN;
    static constexpr int smem_bytes = 1024 + stages * stage_bytes + BAR_BYTES;
    static_assert(smem_bytes <= 227 * 1024, "single-CTA kernel shared memory");
};

template <bool A_MN, bool B_MN, int EPI, int SBN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const KArgs p) {
    using G = SingleGeom<SBN>;
    constexpr int kStages = G::stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * A_TILE_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * G::stage_bytes);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, NUM_EPI_WARPS);
        }
        mbar_init(drain, 1);
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, G::tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Set-up above overlaps the previous launch's tail; no global memory is touched before
    // the previous grid has completed.
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0;        // bit s: stage s has been armed at least once
            uint32_t last_parity = 0;  // bit s: parity of the phase last armed on stage s
            bool ok = true;
            const int k_end = p.kb_per_shard * BK;
            for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
                int mb, nb, shard;
                decode_tile(p, t, mb, nb, shard);
                const int row0 = mb * BM, col0 = nb * SBN;
                // sum mode: the K loop walks (shard, k); batched: shard fixed per tile
                int sa = p.sum_shards ? 0 : (p.a_batched ? shard : 0);
                int sb = p.sum_shards ? 0 : (p.b_batched ? shard : 0);
                int k0 = 0;
                for (int it = 0; it < p.k_iters; ++it) {
                    if (!mbar_wait_bounded(empty + stage, phase ^ 1u, p.status, p.timeout_ns, kWhereProducer)) {
                        ok = false;
                        break;
                    }
                    uint64_t* fb = full + stage;
                    mbar_arrive_expect_tx(fb, G::stage_bytes);
                    armed |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    uint8_t* a_dst = sA + stage * A_TILE_BYTES;
                    uint8_t* b_dst = sB + stage * G::b_bytes;
                    if constexpr (!A_MN) {
                        tma_load_3d(a_dst, &tmA, fb, k0, row0, sa);
                    } else if (p.a_chunked) {
                        tma_load_4d(a_dst, &tmA, fb, 0, k0, row0 / 64, sa);
                    } else {
#pragma unroll
                        for (int c = 0; c < BM / 64; ++c)
                            tma_load_3d(a_dst + c * MN_CHUNK_BYTES, &tmA, fb, row0 + c * 64, k0, sa);
                    }
                    if constexpr (!B_MN) {
                        tma_load_3d(b_dst, &tmB, fb, k0, col0, sb);
                    } else if (p.b_chunked) {
                        tma_load_4d(b_dst, &tmB, fb, 0, k0, col0 / 64, sb);
                    } else {
#pragma unroll
                        for (int c = 0; c < SBN / 64; ++c)
                            tma_load_3d(b_dst + c * MN_CHUNK_BYTES, &tmB, fb, col0 + c * 64, k0, sb);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    k0 += BK;
                    if (k0 == k_end) {  // next shard of the sum (only reached mid-tile in sum mode)
                        k0 = 0;
                        ++sa;
                        ++sb;
                    }
                }
            }
            if (!ok) {
                // Let every copy already issued land before the CTA can exit.
                for (int s = 0; s < kStages; ++s)
                    if (armed & (1u << s))
                        mbar_wait_bounded(full + s, (last_parity >> s) & 1u, p.status, p.timeout_ns, kWhereDrain,
                                          /*watch_status=*/false);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(BM, SBN, A_MN, B_MN);
            const uint64_t a_desc0 = A_MN ? sdesc_sw128(smem_u32(sA), TPMLP_MN_LBO_BYTES, TPMLP_MN_SBO_BYTES)
                                          : sdesc_sw128(smem_u32(sA), 16, 1024);
            const uint64_t b_desc0 = B_MN ? sdesc_sw128(smem_u32(sB), TPMLP_MN_LBO_BYTES, TPMLP_MN_SBO_BYTES)
                                          : sdesc_sw128(smem_u32(sB), 16, 1024);
            constexpr uint64_t a_kstep = A_MN ? (2048 >> 4) : (32 >> 4);  // one UMMA K step (16 elements)
            constexpr uint64_t b_kstep = B_MN ? (2048 >> 4) : (32 >> 4);
            int stage = 0;
            uint32_t phase = 0;
            int lt = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++lt) {
                const int acc = lt & 1;
                const uint32_t acc_phase = (lt >> 1) & 1;
                if (!mbar_wait_bounded(tempty + acc, acc_phase ^ 1u, p.status, p.timeout_ns, kWhereMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * SBN;
                for (int it = 0; it < p.k_iters; ++it) {
                    if (!mbar_wait_bounded(full + stage, phase, p.status, p.timeout_ns, kWhereMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptor start addresses are in 16-byte units in the low bits
                    const uint64_t adesc = a_desc0 + static_cast<uint64_t>(stage * (A_TILE_BYTES >> 4));
                    const uint64_t bdesc = b_desc0 + static_cast<uint64_t>(stage * (G::b_bytes >> 4));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_f16(d_tmem, adesc + kk * a_kstep, bdesc + kk * b_kstep, idesc, (it | kk) != 0 ? 1u : 0u);
                    umma_commit(empty + stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) umma_commit(tfull + acc);
            }
            // Every UMMA issued by this thread has completed once `drain` flips.
            umma_commit(drain);
            mbar_wait_bounded(drain, 0, p.status, p.timeout_ns, kWhereDrain, /*watch_status=*/false);
        }
    } else if (warp >= FIRST_EPI_WARP) {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;                        // TMEM lane quarter of this warp
        const int half = (warp - FIRST_EPI_WARP) >> 2;  // column half of the tile
        int lt = 0;
        for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++lt) {
            const int acc = lt & 1;
            const uint32_t acc_phase = (lt >> 1) & 1;
            if constexpr (EPI == EPI_DGELU) {
                // the tile's first H chunk loads while the accumulator is being computed
                int mb, nb, shard;
                decode_tile(p, t, mb, nb, shard);
                const int gm = mb * BM + q * 32 + lane;
                uint32_t h0[16], h1[16];
                load_h_raw(p, gm, nb * SBN + half * (SBN / 2), shard, h0);
                int okw = 0;
                if (lane == 0) okw = mbar_wait_bounded(tfull + acc, acc_phase, p.status, p.timeout_ns, kWhereEpilogue);
                okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
                if (!okw) break;
                tc_fence_after();
                const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * SBN;
                dgelu_chunks<SBN / 64, SBN>(p, t_row, gm, nb, half * (SBN / 64), shard, h0, h1);
            } else {
            int okw = 0;
            if (lane == 0) okw = mbar_wait_bounded(tfull + acc, acc_phase, p.status, p.timeout_ns, kWhereEpilogue);
            okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
            if (!okw) break;
            tc_fence_after();
            int mb, nb, shard;
            decode_tile(p, t, mb, nb, shard);
            const int gm = mb * BM + q * 32 + lane;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * SBN;
            epilogue_tile<EPI, SBN / 64>(p, t_row, gm, nb, half, shard);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty + acc);
        }
    }

    __syncwarp();  // reconverge the single-lane producer / MMA branches
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, G::tmem_cols);
    }
}


// ---------------------------------------------------------------------------
// Staged epilogue (CTA-pair kernel, short K loops): through shared memory and TMA
// stores.
//
// Each epilogue warp owns a 4 KiB staging buffer.  Per 32-column chunk its 32
// threads (one output row each) write the converted values into a 32-row box in
// the layout a swizzled TMA store expects, and lane 0 stores the box with one
// cp.async.bulk.tensor (the tensor map clips rows >= M and columns >= N):
//   bf16 box: 32 rows x 64 B, 64-byte swizzle: 16-byte chunk c of row r at c ^ ((r >> 1) & 3)
//   fp32 box: 32 rows x 128 B, 128-byte swizzle: chunk c of row r at c ^ (r & 7)
// Both patterns spread the 32 rows of one warp store over all banks.  Such an
// epilogue finishes a 256x256 tile in well under half the time of per-row 16-byte
// global stores (which touch 32 L2 lines per warp instruction), but moves every
// output byte through shared memory twice, which slows a concurrent main loop
// per clock; it is the faster choice when the K loop of a tile is short and the
// epilogue, not the main loop, would set the pace.
// ---------------------------------------------------------------------------
constexpr int EPI_WARP_BYTES = 4096;

__device__ __forceinline__ void stage_bf16x32(uint8_t* box, int r, const float* v) {
    uint8_t* row = box + r * 64;
    const int sw = (r >> 1) & 3;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4 u;
        u.x = pack_bf16x2(v[8 * c + 0], v[8 * c + 1]);
        u.y = pack_bf16x2(v[8 * c + 2], v[8 * c + 3]);
        u.z = pack_bf16x2(v[8 * c + 4], v[8 * c + 5]);
        u.w = pack_bf16x2(v[8 * c + 6], v[8 * c + 7]);
        *reinterpret_cast<uint4*>(row + ((c ^ sw) << 4)) = u;
    }
}
__device__ __forceinline__ void stage_f32x32(uint8_t* box, int r, const float* v) {
    uint8_t* row = box + r * 128;
    const int sw = r & 7;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(row + ((c ^ sw) << 4)) =
            make_float4(v[4 * c + 0], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

// Staged epilogue of one warp's 32 rows x 128 columns of a tile (EPI_BIAS_ACT, EPI_DGELU,
// EPI_STORE).  row0 = the warp's first output row, lane = its row within the box; seq
// counts the warp's staged chunks across tiles, so that consecutive chunks of a single
// bf16 output always alternate between the two 2 KiB boxes.
template <int EPI>
__device__ __forceinline__ void epilogue_tile_staged(const KArgs& p, const CUtensorMap* tm_out,
                                                     const CUtensorMap* tm_out2, uint32_t t_row, int row0, int lane,
                                                     int nb, int half, int shard, uint8_t* ebuf, uint32_t& seq) {
    if (row0 >= p.M) return;
    const bool two = (EPI == EPI_BIAS_ACT) && p.out2 != nullptr;  // Y and the pre-activation H
    const bool f32 = (EPI == EPI_STORE) && p.out_f32;
    const bool one_buffer = two || f32;  // 4 KiB per chunk; otherwise two 2 KiB boxes alternate
    const int gm = row0 + lane;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        const int col = half * 128 + c * 32;
        const int gn0 = nb * BN + col;
        if (gn0 >= p.N) break;
        const int nvalid = p.N - gn0;
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + col, r);
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        uint8_t* box = one_buffer ? ebuf : ebuf + (seq & 1u) * 2048;
        ++seq;
        // the box may be rewritten once the TMA engine has read its previous contents
        // (single output: that was the chunk before last, so one group may stay pending)
        if (lane == 0) {
            if (one_buffer) bulk_wait_group_read<0>();
            else bulk_wait_group_read<1>();
        }
        __syncwarp();
        if constexpr (EPI == EPI_BIAS_ACT) {
            if (p.bias != nullptr) {
                const __nv_bfloat16* bp = static_cast<const __nv_bfloat16*>(p.bias) + shard * p.bias_ss + gn0;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    if (g * 8 < nvalid) {
                        float bf[8];
                        unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(bp + g * 8)), bf);
#pragma unroll
                        for (int i = 0; i < 8; i += 2)
                            f2_unpack(f2_add(f2_pack(v[g * 8 + i], v[g * 8 + i + 1]), f2_pack(bf[i], bf[i + 1])),
                                      v[g * 8 + i], v[g * 8 + i + 1]);
                    }
                }
            }
            if (two) stage_bf16x32(ebuf + 2048, lane, v);
            if (p.act == TPMLP_ACT_GELU_ERF) gelu_inplace32(v);
            stage_bf16x32(box, lane, v);
        } else if constexpr (EPI == EPI_DGELU) {
            if (gm < p.M) {
                const __nv_bfloat16* hp =
                    static_cast<const __nv_bfloat16*>(p.aux) + shard * p.aux_ss + (long long)gm * p.aux_ld + gn0;
                float hv[32];
                load_bf16x32(hp, hv, nvalid, p.st32);
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    if (g * 8 < nvalid) dgelu_mul8(v + g * 8, hv + g * 8);
            }
            stage_bf16x32(box, lane, v);
        } else {
            if (f32) stage_f32x32(box, lane, v);
            else stage_bf16x32(box, lane, v);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(tm_out, box, gn0, row0, shard);
            if (two) tma_store_3d(tm_out2, ebuf + 2048, gn0, row0, shard);
            bulk_commit_group();
        }
    }
}

// Staged GeLU' epilogue of one warp's 32 rows x 128 columns (column half `half`), with each
// chunk's H loaded one chunk ahead (h0 holds the first chunk's on entry): the same values and
// boxes as epilogue_tile_staged<EPI_DGELU>.
__device__ __forceinline__ void epilogue_tile_staged_dgelu(const KArgs& p, const CUtensorMap* tm_out, uint32_t t_row,
                                                           int row0, int lane, int nb, int half, int shard,
                                                           uint8_t* ebuf, uint32_t& seq, uint32_t (&h0)[16],
                                                           uint32_t (&h1)[16]) {
    if (row0 >= p.M) return;
    const int gm = row0 + lane;
#pragma unroll 1
    for (int c = 0; c < 4; c += 2) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            uint32_t(&cur)[16] = k == 0 ? h0 : h1;
            uint32_t(&nxt)[16] = k == 0 ? h1 : h0;
            const int col = half * 128 + (c + k) * 32;
            const int gn0 = nb * BN + col;
            if (gn0 >= p.N) return;
            if (c + k + 1 < 4) load_h_raw(p, gm, gn0 + 32, shard, nxt);
            const int nvalid = p.N - gn0;
            uint32_t r[32];
            tmem_ld_32x32b_x32(t_row + col, r);
            tmem_ld_wait();
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
            uint8_t* box = ebuf + (seq & 1u) * 2048;  // two 2 KiB boxes alternate (single bf16 output)
            ++seq;
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            if (gm < p.M) dgelu_apply32(v, cur, nvalid);
            stage_bf16x32(box, lane, v);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(tm_out, box, gn0, row0, shard);
                bulk_commit_group();
            }
        }
    }
}

// ============================================================================
// CTA-pair variant: a cluster of two CTAs on neighbouring SMs computes one
// 256x256 output tile with tcgen05.mma.cta_group::2 (M=256, N=256, K=16).
// CTA r (r = %cluster_ctarank) loads rows [256 mb + 128 r, +128) of A and
// columns [256 nb + 128 r, +128) of B into its own shared memory; the UMMA
// reads A from each CTA and exchanges the B halves in hardware, and writes
// rows 128 r .. 128 r + 127 of the tile into CTA r's tensor memory.  So each
// SM holds half as many B bytes per stage as the single-CTA kernel (32 KiB
// stages, seven in flight) and the pair reads a third fewer bytes from L2.
//
//   leader (r = 0)  warp 0: TMA producer, arms its full barrier for both CTAs'
//                            bytes (the peer's copies complete on it too)
//                   warp 1: UMMA issuer; commits multicast to both CTAs'
//                            empty / tmem-full barriers
//   peer   (r = 1)  warp 0: TMA producer (gated by its own empty barrier)
//   both            warp 1: TMEM allocation (collective for the pair)
//                   warps 4-11 (4-7): epilogue of its 128 rows; the accumulator
//                            is released by 16 (8) arrivals on the leader's barrier
//
// Every TMA load lands in the issuing CTA's own shared memory (no multicast):
// the library may run on every GPU of a multi-GPU job, and each operand byte is
// already read once per pair.
// ============================================================================
constexpr int P_A_BYTES = BM * BK * 2;        // 16 KiB: this CTA's 128 rows of A
constexpr int P_B_BYTES = (BN / 2) * BK * 2;  // 16 KiB: this CTA's 128 columns of B
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;

// STAGED = false: direct-store epilogue, 7 stages.  STAGED = true: staged (TMA-store)
// epilogue, 6 stages + 8 x 4 KiB staging boxes.
//
// Epilogue warps: the staged epilogue (short K loops, where the epilogue sets the pace) runs
// on 8 warps, two per TMEM lane quarter, each taking one 128-column half of the tile; the
// direct-store epilogue runs on 4, one per lane quarter, each taking both halves in turn.
// Its work per tile is the same, spread over twice the time behind a K loop long enough to
// hide it, and the main loop it overlaps runs ~1 % faster at the power cap (interleaved A/B
// of the fwd+bwd step, bit-identical results): fewer concurrent epilogue warps leave more of
// the SM's issue slots and load/store data path to the producer and the UMMA issuer.
template <bool STAGED>
struct PairGeom {
    static constexpr int epi_warps = STAGED ? NUM_EPI_WARPS : 4;
    static constexpr int threads = 32 * (FIRST_EPI_WARP + epi_warps);
    static constexpr int stages = STAGED ? 6 : 7;
    static constexpr int epi_bytes = STAGED ? NUM_EPI_WARPS * EPI_WARP_BYTES : 0;
    static constexpr int smem_bytes = 1024 + stages * P_STAGE_BYTES + epi_bytes + BAR_BYTES;
    static_assert(smem_bytes <= 227 * 1024, "pair kernel shared memory");
};

template <bool A_MN, bool B_MN, int EPI, bool STAGED>
__global__ void __launch_bounds__(PairGeom<STAGED>::threads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmO2,
                     const KArgs p) {
    constexpr int P_STAGES = PairGeom<STAGED>::stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + P_STAGES * P_A_BYTES;
    uint8_t* sE = smem + P_STAGES * P_STAGE_BYTES;  // staging boxes (STAGED), 1 KiB aligned
    uint64_t* full = reinterpret_cast<uint64_t*>(sE + PairGeom<STAGED>::epi_bytes);
    uint64_t* empty = full + P_STAGES;
    uint64_t* tfull = empty + P_STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t prank = cluster_ctarank();  // position in the CTA pair
    const uint32_t pleader = 0;                // the pair's leader (UMMA issuer)
    const bool leader = prank == 0;
    const uint16_t pair_mask = 0x3;
    const int cluster_id = blockIdx.x / 2;
    const int n_clusters = gridDim.x / 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, 2 * PairGeom<STAGED>::epi_warps);
        }
        mbar_init(drain, 1);
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if constexpr (STAGED) {
        if (warp == FIRST_EPI_WARP && lane == 0) {
            tma_prefetch_desc(&tmO);
            tma_prefetch_desc(&tmO2);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer may signal the leader's barriers from here on
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Set-up above overlaps the previous launch's tail; no global memory is touched before
    // the previous grid has completed.
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, last_parity = 0;
            bool ok = true;
            const int k_end = p.kb_per_shard * BK;
            const uint32_t full_leader0 = mapa_shared(smem_u32(full), pleader);  // the pair leader's barriers
            for (int t = p.tile_begin + cluster_id; t < p.num_tiles && ok; t += n_clusters) {
                int mb, nb, shard;
                decode_tile(p, t, mb, nb, shard);
                const int row0 = mb * (2 * BM) + static_cast<int>(prank) * BM;
                const int col0 = nb * BN + static_cast<int>(prank) * (BN / 2);
                // Odd waves walk K backwards: a tile of the next wave usually shares its
                // A (or B) panel with a tile of this one, and starts on the K range that
                // this wave read last and the L2 still holds.  Waves are counted as those
                // of the full grid (rev_period tiles each), so a tile's accumulation order,
                // and its bits, do not depend on the grid it runs on.
                const bool rev = ((t / p.rev_period) & 1) != 0;
                int sa = p.sum_shards ? (rev ? p.n_shards - 1 : 0) : (p.a_batched ? shard : 0);
                int sb = p.sum_shards ? (rev ? p.n_shards - 1 : 0) : (p.b_batched ? shard : 0);
                int k0 = rev ? k_end - BK : 0;
                for (int it = 0; it < p.k_iters; ++it) {
                    if (!mbar_wait_bounded(empty + stage, phase ^ 1u, p.status, p.timeout_ns, kWhereProducer)) {
                        ok = false;
                        break;
                    }
                    if (leader) {
                        mbar_arrive_expect_tx(full + stage, 2 * P_STAGE_BYTES);
                        armed |= 1u << stage;
                        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    }
                    const uint32_t bar = full_leader0 + stage * 8;
                    uint8_t* a_dst = sA + stage * P_A_BYTES;
                    uint8_t* b_dst = sB + stage * P_B_BYTES;
                    if constexpr (!A_MN) {
                        tma_load_3d_pair(a_dst, &tmA, bar, k0, row0, sa);
                    } else if (p.a_chunked) {
                        tma_load_4d_pair(a_dst, &tmA, bar, 0, k0, row0 / 64, sa);
                    } else {
#pragma unroll
                        for (int c = 0; c < BM / 64; ++c)
                            tma_load_3d_pair(a_dst + c * MN_CHUNK_BYTES, &tmA, bar, row0 + c * 64, k0, sa);
                    }
                    if constexpr (!B_MN) {
                        tma_load_3d_pair(b_dst, &tmB, bar, k0, col0, sb);
                    } else if (p.b_chunked) {
                        tma_load_4d_pair(b_dst, &tmB, bar, 0, k0, col0 / 64, sb);
                    } else {
#pragma unroll
                        for (int c = 0; c < (BN / 2) / 64; ++c)
                            tma_load_3d_pair(b_dst + c * MN_CHUNK_BYTES, &tmB, bar, col0 + c * 64, k0, sb);
                    }
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (!rev) {
                        k0 += BK;
                        if (k0 == k_end) {
                            k0 = 0;
                            ++sa;
                            ++sb;
                        }
                    } else {
                        k0 -= BK;
                        if (k0 < 0) {
                            k0 = k_end - BK;
                            --sa;
                            --sb;
                        }
                    }
                }
            }
            if (ok) {
                // The UMMA commits that release stages arrive on this CTA's empty barriers from
                // the pair leader, possibly on the other SM, and nothing else orders them
                // before the cluster's final barrier: wait for the release of every stage's last
                // use, so that no arrival can reach this CTA's shared memory after it exits.
                for (int i = 0; i < P_STAGES; ++i) {
                    if (!mbar_wait_bounded(empty + stage, phase ^ 1u, p.status, p.timeout_ns, kWhereDrain)) break;
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (leader) {
                    // the leader's full barriers count both CTAs' copies: wait for all of them
                    for (int s = 0; s < P_STAGES; ++s)
                        if (armed & (1u << s))
                            mbar_wait_bounded(full + s, (last_parity >> s) & 1u, p.status, p.timeout_ns, kWhereDrain,
                                              /*watch_status=*/false);
                }
                // let this CTA's last copies (counted on the leader's barriers) land before
                // either CTA of the pair can exit
                if (!leader) spin_ns(200000);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            if (leader) {
                // -------------------------------------------------------- UMMA issuer (leader)
                constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN, A_MN, B_MN);
                const uint64_t a_desc0 = A_MN ? sdesc_sw128(smem_u32(sA), TPMLP_MN_LBO_BYTES, TPMLP_MN_SBO_BYTES)
                                              : sdesc_sw128(smem_u32(sA), 16, 1024);
                const uint64_t b_desc0 = B_MN ? sdesc_sw128(smem_u32(sB), TPMLP_MN_LBO_BYTES, TPMLP_MN_SBO_BYTES)
                                              : sdesc_sw128(smem_u32(sB), 16, 1024);
                constexpr uint64_t a_kstep = A_MN ? (2048 >> 4) : (32 >> 4);
                constexpr uint64_t b_kstep = B_MN ? (2048 >> 4) : (32 >> 4);
                int stage = 0;
                uint32_t phase = 0;
                int lt = 0;
                bool ok = true;
                for (int t = p.tile_begin + cluster_id; t < p.num_tiles && ok; t += n_clusters, ++lt) {
                    const int acc = lt & 1;
                    const uint32_t acc_phase = (lt >> 1) & 1;
                    if (!mbar_wait_bounded(tempty + acc, acc_phase ^ 1u, p.status, p.timeout_ns, kWhereMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * BN;
                    for (int it = 0; it < p.k_iters; ++it) {
                        if (!mbar_wait_bounded(full + stage, phase, p.status, p.timeout_ns, kWhereMma)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t adesc = a_desc0 + static_cast<uint64_t>(stage * (P_A_BYTES >> 4));
                        const uint64_t bdesc = b_desc0 + static_cast<uint64_t>(stage * (P_B_BYTES >> 4));
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            umma_f16_pair(d_tmem, adesc + kk * a_kstep, bdesc + kk * b_kstep, idesc,
                                          (it | kk) != 0 ? 1u : 0u);
                        // the stage is free for the producers of both CTAs
                        umma_commit_pair_mc(empty + stage, pair_mask);
                        if (++stage == P_STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok) umma_commit_pair_mc(tfull + acc, pair_mask);
                }
                umma_commit_pair_mc(drain, pair_mask);
                // both accumulators' last releases (16 epilogue warps of the pair, half of them
                // arriving from the peer SM) land before this CTA can exit
                for (int i = 0; ok && i < 2; ++i, ++lt)
                    ok = mbar_wait_bounded(tempty + (lt & 1), ((lt >> 1) & 1) ^ 1u, p.status, p.timeout_ns, kWhereDrain);
            }
            // both CTAs: every UMMA (and its commit arrivals) is done once `drain` flips
            mbar_wait_bounded(drain, 0, p.status, p.timeout_ns, kWhereDrain, /*watch_status=*/false);
        }
    } else if (warp >= FIRST_EPI_WARP) {
        // ---------------------------------------------------------------- epilogue (both CTAs)
        const int q = warp & 3;
        [[maybe_unused]] const int half = (warp - FIRST_EPI_WARP) >> 2;  // STAGED only
        const uint32_t tempty_leader0 = mapa_shared(smem_u32(tempty), pleader);
        [[maybe_unused]] uint8_t* ebuf = sE + (warp - FIRST_EPI_WARP) * EPI_WARP_BYTES;  // STAGED only
        uint32_t seq = 0;
        int lt = 0;
        for (int t = p.tile_begin + cluster_id; t < p.num_tiles; t += n_clusters, ++lt) {
            const int acc = lt & 1;
            const uint32_t acc_phase = (lt >> 1) & 1;
            if constexpr (EPI == EPI_DGELU) {
                // the tile's first H chunk loads while the accumulator is being computed
                int mb, nb, shard;
                decode_tile(p, t, mb, nb, shard);
                const int row0 = mb * (2 * BM) + static_cast<int>(prank) * BM + q * 32;
                uint32_t h0[16], h1[16];
                load_h_raw(p, row0 + lane, nb * BN + (STAGED ? half * 128 : 0), shard, h0);
                int okw = 0;
                if (lane == 0) okw = mbar_wait_bounded(tfull + acc, acc_phase, p.status, p.timeout_ns, kWhereEpilogue);
                okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
                if (!okw) break;
                tc_fence_after();
                const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
                if constexpr (STAGED)
                    epilogue_tile_staged_dgelu(p, &tmO, t_row, row0, lane, nb, half, shard, ebuf, seq, h0, h1);
                else
                    dgelu_chunks<8, BN>(p, t_row, row0 + lane, nb, 0, shard, h0, h1);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_leader0 + acc * 8);
                continue;
            }
            int okw = 0;
            if (lane == 0) okw = mbar_wait_bounded(tfull + acc, acc_phase, p.status, p.timeout_ns, kWhereEpilogue);
            okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
            if (!okw) break;
            tc_fence_after();
            int mb, nb, shard;
            decode_tile(p, t, mb, nb, shard);
            const int row0 = mb * (2 * BM) + static_cast<int>(prank) * BM + q * 32;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            if constexpr (STAGED) {
                epilogue_tile_staged<EPI>(p, &tmO, &tmO2, t_row, row0, lane, nb, half, shard, ebuf, seq);
            } else {
                static_assert(STAGED || PairGeom<STAGED>::epi_warps == 4, "direct epilogue: one warp per lane quarter");
                epilogue_tile<EPI>(p, t_row, row0 + lane, nb, 0, shard);
                epilogue_tile<EPI>(p, t_row, row0 + lane, nb, 1, shard);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader0 + acc * 8);
        }
        if constexpr (STAGED) {
            if (lane == 0) bulk_wait_group_all();  // this warp's output stores are complete
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no CTA leaves while its peer may still touch its shared or tensor memory
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}


// ============================================================================
// Split-K CTA pairs, for shard-summing GEMMs (the row layer's Z = sum_i Y_i B_i and the
// backward's dX = sum_i dH_i A_i^T) whose 256x256 tiles are fewer than the CTA pairs the
// GPU holds.  Such GEMMs otherwise run on 128x128 single-CTA tiles, whose main loop is
// bound by each SM's operand bandwidth (32 KiB per 256 tensor cycles).
//
// A cluster of four CTAs -- two CTA pairs -- computes one 256x256 output tile; pair
// q = rank / 2 accumulates K blocks [q kh, ...) of the tile's K loop (kh = k_iters / 2)
// into its own tensor memory with the same producer / UMMA structure as gemm_pair_kernel
// (32 KiB per 512 tensor cycles per SM).  The two fp32 partial sums meet in distributed
// shared memory: CTA (q, r) finishes column half q of its 128 rows, so once the partner
// CTA (1 - q, r) -- same rows, other K half -- reports that its own products are complete
// (its operand ring is then free), it writes the other column half of its partial
// (128 x 128 fp32) into the partner's ring, and receives the matching half in its own.
// The thread that holds a row in one CTA reads it back in the other (same lane quarter and
// lane), so the buffer is laid out by thread: 16-byte piece j of thread x's row at slot
// j * 128 + x, and each warp store or load covers 512 contiguous bytes.
// Each CTA adds the two partials and runs the usual epilogue on its half.  Every TMA load
// lands in the CTA that issues it (no multicast); every wait is bounded.
//
// One tile per cluster: the host launches 4 * (num_tiles - tile_begin) CTAs.  Also used for the
// last partial wave of a multi-wave GEMM, whose full waves run on gemm_pair_kernel.
// ============================================================================
constexpr int SK_THREADS = 256;     // warp 0 producer, warp 1 TMEM + UMMA issuer, warps 4-7 epilogue
constexpr int SK_STAGES = 7;
constexpr int SK_SMEM = 1024 + SK_STAGES * P_STAGE_BYTES + BAR_BYTES;
static_assert(BM * 128 * 4 <= SK_STAGES * P_A_BYTES, "the received half fits in the A ring");
static_assert(SK_SMEM <= 227 * 1024, "split-K kernel shared memory");

template <bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(SK_THREADS, 1)
    gemm_splitk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const KArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + SK_STAGES * P_A_BYTES;
    uint4* recv = reinterpret_cast<uint4*>(smem);  // 32 x 128 16-byte slots, over the A ring once it is free
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SK_STAGES * P_STAGE_BYTES);
    uint64_t* empty = full + SK_STAGES;
    uint64_t* tfull = empty + SK_STAGES;
    uint64_t* drain = tfull + 1;
    uint64_t* peer_free = drain + 1;   // the partner's products are complete (one arrival per epilogue warp)
    uint64_t* data_ready = peer_free + 1;  // the partner's half has landed in recv (one per epilogue thread)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(data_ready + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t prank = rank & 1u;     // position in the CTA pair
    const uint32_t pleader = rank & ~1u;  // the pair's leader (UMMA issuer)
    const int q = static_cast<int>(rank >> 1);  // the K half this pair accumulates, and the column half it finishes
    const bool leader = prank == 0;
    const uint16_t pair_mask = static_cast<uint16_t>(0x3u << pleader);
    const uint32_t partner = rank ^ 2u;   // same rows, other K half
    const int t = p.tile_begin + static_cast<int>(blockIdx.x) / 4;
    const int kh = p.k_iters / 2;
    const int it0 = q ? kh : 0, it1 = q ? p.k_iters : kh;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SK_STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(tfull, 1);
        mbar_init(drain, 1);
        mbar_init(peer_free, 4);
        mbar_init(data_ready, 128);
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, BN);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // every barrier of the cluster is initialised from here on
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch_dependents();

    int mb, nb, shard;
    decode_tile(p, t, mb, nb, shard);

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ producer (all four CTAs)
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, last_parity = 0;
            bool ok = true;
            const int k_end = p.kb_per_shard * BK;
            const uint32_t full_leader0 = mapa_shared(smem_u32(full), pleader);
            const int row0 = mb * (2 * BM) + static_cast<int>(prank) * BM;
            const int col0 = nb * BN + static_cast<int>(prank) * (BN / 2);
            int sa, sb, k0;
            if (p.sum_shards) {
                sa = sb = it0 / p.kb_per_shard;
                k0 = (it0 - sa * p.kb_per_shard) * BK;
            } else {
                sa = p.a_batched ? shard : 0;
                sb = p.b_batched ? shard : 0;
                k0 = it0 * BK;
            }
            for (int it = it0; it < it1; ++it) {
                if (!mbar_wait_bounded(empty + stage, phase ^ 1u, p.status, p.timeout_ns, kWhereProducer)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    mbar_arrive_expect_tx(full + stage, 2 * P_STAGE_BYTES);
                    armed |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                }
                const uint32_t bar = full_leader0 + stage * 8;
                uint8_t* a_dst = sA + stage * P_A_BYTES;
                uint8_t* b_dst = sB + stage * P_B_BYTES;
                if constexpr (!A_MN) {
                    tma_load_3d_pair(a_dst, &tmA, bar, k0, row0, sa);
                } else if (p.a_chunked) {
                    tma_load_4d_pair(a_dst, &tmA, bar, 0, k0, row0 / 64, sa);
                } else {
#pragma unroll
                    for (int c = 0; c < BM / 64; ++c)
                        tma_load_3d_pair(a_dst + c * MN_CHUNK_BYTES, &tmA, bar, row0 + c * 64, k0, sa);
                }
                if constexpr (!B_MN) {
                    tma_load_3d_pair(b_dst, &tmB, bar, k0, col0, sb);
                } else if (p.b_chunked) {
                    tma_load_4d_pair(b_dst, &tmB, bar, 0, k0, col0 / 64, sb);
                } else {
#pragma unroll
                    for (int c = 0; c < (BN / 2) / 64; ++c)
                        tma_load_3d_pair(b_dst + c * MN_CHUNK_BYTES, &tmB, bar, col0 + c * 64, k0, sb);
                }
                if (++stage == SK_STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
                k0 += BK;
                if (k0 == k_end) {  // next shard of the sum
                    k0 = 0;
                    ++sa;
                    ++sb;
                }
            }
            if (ok) {
                // the leader's commits that release stages arrive on this CTA's empty barriers,
                // possibly from the other SM of the pair: observe each stage's last release
                for (int i = 0; i < SK_STAGES; ++i) {
                    if (!mbar_wait_bounded(empty + stage, phase ^ 1u, p.status, p.timeout_ns, kWhereDrain)) break;
                    if (++stage == SK_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            } else {
                if (leader) {
                    for (int s = 0; s < SK_STAGES; ++s)
                        if (armed & (1u << s))
                            mbar_wait_bounded(full + s, (last_parity >> s) & 1u, p.status, p.timeout_ns, kWhereDrain,
                                              /*watch_status=*/false);
                } else {
                    spin_ns(200000);  // let this CTA's last copies (counted on the leader's barriers) land
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            if (leader) {
                // -------------------------------------------------------- UMMA issuer (pair leaders)
                constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN, A_MN, B_MN);
                const uint64_t a_desc0 = A_MN ? sdesc_sw128(smem_u32(sA), TPMLP_MN_LBO_BYTES, TPMLP_MN_SBO_BYTES)
                                              : sdesc_sw128(smem_u32(sA), 16, 1024);
                const uint64_t b_desc0 = B_MN ? sdesc_sw128(smem_u32(sB), TPMLP_MN_LBO_BYTES, TPMLP_MN_SBO_BYTES)
                                              : sdesc_sw128(smem_u32(sB), 16, 1024);
                constexpr uint64_t a_kstep = A_MN ? (2048 >> 4) : (32 >> 4);
                constexpr uint64_t b_kstep = B_MN ? (2048 >> 4) : (32 >> 4);
                int stage = 0;
                uint32_t phase = 0;
                bool ok = true;
                for (int i = 0; i < it1 - it0; ++i) {
                    if (!mbar_wait_bounded(full + stage, phase, p.status, p.timeout_ns, kWhereMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = a_desc0 + static_cast<uint64_t>(stage * (P_A_BYTES >> 4));
                    const uint64_t bdesc = b_desc0 + static_cast<uint64_t>(stage * (P_B_BYTES >> 4));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_f16_pair(tmem_base, adesc + kk * a_kstep, bdesc + kk * b_kstep, idesc,
                                      (i | kk) != 0 ? 1u : 0u);
                    umma_commit_pair_mc(empty + stage, pair_mask);
                    if (++stage == SK_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) umma_commit_pair_mc(tfull, pair_mask);
                umma_commit_pair_mc(drain, pair_mask);
            }
            mbar_wait_bounded(drain, 0, p.status, p.timeout_ns, kWhereDrain, /*watch_status=*/false);
        }
    } else if (warp >= FIRST_EPI_WARP) {
        // ---------------------------------------------------------------- exchange + epilogue
        const int ql = warp & 3;             // TMEM lane quarter
        const int row_l = ql * 32 + lane;    // this thread's row among the CTA's 128
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(ql * 32) << 16);
        int okw = 0;
        if (lane == 0) okw = mbar_wait_bounded(tfull, 0, p.status, p.timeout_ns, kWhereEpilogue);
        okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
        if (okw) {
            tc_fence_after();
            // this CTA's products are complete: its A ring may take the partner's half
            fence_proxy_async_all();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(peer_free), partner));
            // every lane acquires the partner's release itself: its own writes follow
            const bool okp = __all_sync(0xFFFFFFFFu,
                                        mbar_wait_bounded_cluster(peer_free, 0, p.status, p.timeout_ns, kWhereExchange));
            if (okp) {
                // the other column half of this CTA's partial, into the partner's ring
                const uint32_t dst = mapa_shared(smem_u32(recv + row_l), partner);
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + (1 - q) * 128 + c * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_cluster_v4(dst + ((c * 8 + j) * 128) * 16, r[4 * j], r[4 * j + 1], r[4 * j + 2],
                                      r[4 * j + 3]);
                }
                mbar_arrive_cluster(mapa_shared(smem_u32(data_ready), partner));
                // every lane acquires: each reads rows the partner's threads wrote
                const bool okd = __all_sync(
                    0xFFFFFFFFu, mbar_wait_bounded_cluster(data_ready, 0, p.status, p.timeout_ns, kWhereExchange));
                if (okd) {
                    // own half: this CTA's partial plus the partner's, then the usual epilogue
                    const int gm = mb * (2 * BM) + static_cast<int>(prank) * BM + row_l;
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        const int col = q * 128 + c * 32;
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(t_row + col, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint4 u = recv[(c * 8 + j) * 128 + row_l];
                            r[4 * j + 0] = __float_as_uint(__uint_as_float(r[4 * j + 0]) + __uint_as_float(u.x));
                            r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + __uint_as_float(u.y));
                            r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + __uint_as_float(u.z));
                            r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + __uint_as_float(u.w));
                        }
                        epilogue_chunk<EPI>(p, r, gm, nb * BN + col, shard);
                    }
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no CTA leaves while another may still write its shared memory or barriers
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc_pair(tmem_base, BN);
    }
}

}  // namespace tc
}  // namespace tpmlp

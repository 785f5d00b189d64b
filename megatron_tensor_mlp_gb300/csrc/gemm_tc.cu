// Host side of the tcgen05 GEMM: tensor-map encoding, tile geometry, launch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gemm_tc.cuh"
#include "internal.h"

namespace tpmlp {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D bf16 tensor map over [shards][outer][inner] with a (box_inner x box_outer x 1) box, 128-byte swizzle.
bool make_map(CUtensorMap* map, const Operand& op, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    const uint64_t shards = op.shards > 0 ? static_cast<uint64_t>(op.shards) : 1;
    cuuint64_t dims[3] = {inner, outer, shards};
    const uint64_t ld_bytes = static_cast<uint64_t>(op.ld) * 2;
    uint64_t ss_bytes = static_cast<uint64_t>(op.ss) * 2;
    if (shards == 1) ss_bytes = ld_bytes * outer;  // unused extent; any valid multiple of 16
    cuuint64_t strides[2] = {ld_bytes, ss_bytes};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(op.ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d): dims %llu x %llu x %llu, strides %llu %llu", static_cast<int>(r),
                  (unsigned long long)inner, (unsigned long long)outer, (unsigned long long)shards,
                  (unsigned long long)ld_bytes, (unsigned long long)ss_bytes);
        return false;
    }
    return true;
}

template <bool A_MN, bool B_MN, int EPI>
tpmlp_status launch_variant(const CUtensorMap& ma, const CUtensorMap& mb, const tc::KArgs& k, int grid,
                            const DeviceInfo& dev, cudaStream_t st) {
    auto kern = tc::gemm_kernel<A_MN, B_MN, EPI>;
    static bool attr_done[64] = {};
    if (dev.device < 64 && !attr_done[dev.device]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::SMEM_BYTES);
        if (e != cudaSuccess) {
            set_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            return TPMLP_ERR_CUDA;
        }
        attr_done[dev.device] = true;
    }
    kern<<<grid, tc::NUM_THREADS, tc::SMEM_BYTES, st>>>(ma, mb, k);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("tcgen05 GEMM launch: %s", cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    return TPMLP_OK;
}

}  // namespace

tpmlp_status launch_tc_gemm(const Operand& a, const Operand& b, const GemmSpec& g, const DeviceInfo& dev,
                            cudaStream_t st) {
    CUtensorMap ma, mb;
    // A: K-major [shards][M][K]; MN-major [shards][K][M].  B: K-major [shards][N][K]; MN-major [shards][K][N].
    bool ok = a.mn_major ? make_map(&ma, a, g.M, g.K, 64, tc::BK) : make_map(&ma, a, g.K, g.M, tc::BK, tc::BM);
    if (!ok) return TPMLP_ERR_CUDA;
    ok = b.mn_major ? make_map(&mb, b, g.N, g.K, 64, tc::BK) : make_map(&mb, b, g.K, g.N, tc::BK, tc::BN);
    if (!ok) return TPMLP_ERR_CUDA;

    tc::KArgs k{};
    k.M = static_cast<int>(g.M);
    k.N = static_cast<int>(g.N);
    k.K = static_cast<int>(g.K);
    k.n_shards = static_cast<int>(g.n_shards);
    k.sum_shards = g.sum_shards ? 1 : 0;
    k.a_batched = g.a_batched ? 1 : 0;
    k.b_batched = g.b_batched ? 1 : 0;
    k.m_blocks = static_cast<int>((g.M + tc::BM - 1) / tc::BM);
    k.n_blocks = static_cast<int>((g.N + tc::BN - 1) / tc::BN);
    k.batch = g.sum_shards ? 1 : k.n_shards;
    k.num_tiles = k.m_blocks * k.n_blocks * k.batch;
    k.kb_per_shard = static_cast<int>((g.K + tc::BK - 1) / tc::BK);
    k.k_iters = g.sum_shards ? k.kb_per_shard * k.n_shards : k.kb_per_shard;
    k.group_m = 16;
    k.act = g.act;
    k.out_f32 = g.out_f32 ? 1 : 0;
    k.out = g.out;
    k.out_ld = g.out_ld;
    k.out_ss = g.out_ss;
    k.out2 = g.out2;
    k.out2_ld = g.out2_ld;
    k.out2_ss = g.out2_ss;
    k.bias = g.bias;
    k.bias_ss = g.bias_ss;
    k.aux = g.aux;
    k.aux_ld = g.aux_ld;
    k.aux_ss = g.aux_ss;
    k.status = dev.status;
    k.timeout_ns = 2000000000ull;  // 2 s per wait
    if (k.num_tiles == 0) return TPMLP_OK;
    const int grid = k.num_tiles < dev.sm_count ? k.num_tiles : dev.sm_count;

    const bool amn = a.mn_major, bmn = b.mn_major;
    if (g.epi == EPI_BIAS_ACT && !amn && bmn) return launch_variant<false, true, EPI_BIAS_ACT>(ma, mb, k, grid, dev, st);
    if (g.epi == EPI_DGELU && !amn && !bmn) return launch_variant<false, false, EPI_DGELU>(ma, mb, k, grid, dev, st);
    if (g.epi == EPI_STORE && amn && bmn) return launch_variant<true, true, EPI_STORE>(ma, mb, k, grid, dev, st);
    if (g.epi == EPI_STORE && !amn && !bmn) return launch_variant<false, false, EPI_STORE>(ma, mb, k, grid, dev, st);
    set_error("internal: no tcgen05 GEMM variant for epi=%d a_mn=%d b_mn=%d", g.epi, (int)amn, (int)bmn);
    return TPMLP_ERR_CUDA;
}

}  // namespace tpmlp

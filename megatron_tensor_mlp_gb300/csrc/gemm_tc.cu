// Host side of the tcgen05 GEMM: tensor-map encoding, tile geometry, launch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
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

// 3-D tensor map over an output [shards][rows][cols] for the staged epilogue's TMA
// stores: 32 x 32 boxes; bf16 rows of a box are 64 B (64-byte swizzle), fp32 rows 128 B
// (128-byte swizzle), matching the staging layout in shared memory.
bool make_out_map(CUtensorMap* map, void* ptr, int64_t ld, int64_t ss, uint64_t cols, uint64_t rows,
                  uint64_t shards, bool f32) {
    auto fn = encode_fn();
    if (!fn) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    const uint64_t es = f32 ? 4 : 2;
    const uint64_t ld_bytes = static_cast<uint64_t>(ld) * es;
    uint64_t ss_bytes = static_cast<uint64_t>(ss) * es;
    if (shards <= 1) {
        shards = 1;
        ss_bytes = ld_bytes * rows;  // unused extent; any valid multiple of 16
    }
    cuuint64_t dims[3] = {cols, rows, shards};
    cuuint64_t strides[2] = {ld_bytes, ss_bytes};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled (output) failed (%d): dims %llu x %llu x %llu, strides %llu %llu",
                  static_cast<int>(r), (unsigned long long)cols, (unsigned long long)rows,
                  (unsigned long long)shards, (unsigned long long)ld_bytes, (unsigned long long)ss_bytes);
        return false;
    }
    return true;
}

// K blocks per tile up to which the pair kernel uses the staged epilogue: a 256x256 tile's
// main loop takes ~512 cycles per 64-wide K block, a direct-store epilogue ~10-20 k cycles.
constexpr int kStagedMaxKBlocks = 40;

// 0 auto, 1 single-CTA, 2 pair, 3 pair + direct stores, 4 pair + TMA stores, 5 auto with split-K forced
std::atomic<int> g_gemm_mode{0};
std::atomic<int> g_group_m{16};  // M-blocks per raster group
// K blocks per launch of a split fp32 contraction (see launch_tc_gemm)
constexpr int kDefaultKChunkBlocks = 4096;
std::atomic<int> g_k_chunk_blocks{kDefaultKChunkBlocks};

template <typename Kern>
bool set_smem_attr(Kern kern, int device, int bytes, bool* done) {
    if (device < 64 && done[device]) return true;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) {
        set_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return false;
    }
    if (device < 64) done[device] = true;
    return true;
}

// 4-D bf16 tensor map of an MN-major operand whose MN extent is a multiple of 64:
// [shards][mn/64 chunks][K][64], so that one box (64 x BK x chunks x 1) lands in
// shared memory as `chunks` consecutive 64-wide MN chunks of BK K-rows.
bool make_map_chunked(CUtensorMap* map, const Operand& op, uint64_t mn, uint64_t k, uint32_t chunks) {
    auto fn = encode_fn();
    if (!fn) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    const uint64_t shards = op.shards > 0 ? static_cast<uint64_t>(op.shards) : 1;
    const uint64_t ld_bytes = static_cast<uint64_t>(op.ld) * 2;
    uint64_t ss_bytes = static_cast<uint64_t>(op.ss) * 2;
    if (shards == 1) ss_bytes = ld_bytes * k;
    cuuint64_t dims[4] = {64, k, mn / 64, shards};
    cuuint64_t strides[3] = {ld_bytes, 128, ss_bytes};
    cuuint32_t box[4] = {64, static_cast<cuuint32_t>(tc::BK), chunks, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(op.ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled (chunked) failed (%d)", static_cast<int>(r));
        return false;
    }
    return true;
}

template <bool A_MN, bool B_MN, int EPI, int SBN>
tpmlp_status launch_single(const CUtensorMap& ma, const CUtensorMap& mb, const tc::KArgs& k, const DeviceInfo& dev,
                           int max_grid, cudaStream_t st) {
    auto kern = tc::gemm_kernel<A_MN, B_MN, EPI, SBN>;
    constexpr int smem = tc::SingleGeom<SBN>::smem_bytes;
    static bool attr_done[64] = {};
    if (!set_smem_attr(kern, dev.device, smem, attr_done)) return TPMLP_ERR_CUDA;
    int grid = k.num_tiles < dev.sm_count ? k.num_tiles : dev.sm_count;
    if (max_grid > 0 && grid > max_grid) grid = max_grid;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(tc::NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddep_wait
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, k);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("tcgen05 GEMM launch: %s", cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    count_launch();
    return TPMLP_OK;
}

// Co-resident CTA pairs (clusters of two) of the pair kernel on this device (0 if it cannot run).
template <bool A_MN, bool B_MN, int EPI, bool STAGED>
int pair_capacity(const DeviceInfo& dev) {
    static int cap[64];
    static bool done[64];
    static bool attr_done[64] = {};
    if (dev.device >= 64) return 0;
    if (done[dev.device]) return cap[dev.device];
    auto kern = tc::gemm_pair_kernel<A_MN, B_MN, EPI, STAGED>;
    constexpr int smem = tc::PairGeom<STAGED>::smem_bytes;
    int n = 0;
    if (set_smem_attr(kern, dev.device, smem, attr_done)) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (dev.sm_count / 2));
        cfg.blockDim = dim3(tc::PairGeom<STAGED>::threads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
        cudaGetLastError();
    }
    cap[dev.device] = n;
    done[dev.device] = true;
    return n;
}

template <bool A_MN, bool B_MN, int EPI, bool STAGED>
tpmlp_status launch_pair(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                         const CUtensorMap& mo2, const tc::KArgs& k, int clusters, cudaStream_t st) {
    auto kern = tc::gemm_pair_kernel<A_MN, B_MN, EPI, STAGED>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(tc::PairGeom<STAGED>::threads);
    cfg.dynamicSmemBytes = tc::PairGeom<STAGED>::smem_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddep_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, mo, mo2, k);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("tcgen05 CTA-pair GEMM launch: %s", cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    count_launch();
    return TPMLP_OK;
}

// Co-resident clusters of the split-K kernel (two CTA pairs each) on this device.
template <bool A_MN, bool B_MN, int EPI>
int splitk_capacity(const DeviceInfo& dev) {
    static int cap[64];
    static bool done[64];
    static bool attr_done[64] = {};
    if (dev.device >= 64) return 0;
    if (done[dev.device]) return cap[dev.device];
    auto kern = tc::gemm_splitk_kernel<A_MN, B_MN, EPI>;
    int n = 0;
    if (set_smem_attr(kern, dev.device, tc::SK_SMEM, attr_done)) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(4 * (dev.sm_count / 4));
        cfg.blockDim = dim3(tc::SK_THREADS);
        cfg.dynamicSmemBytes = tc::SK_SMEM;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 4;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
        cudaGetLastError();
    }
    cap[dev.device] = n;
    done[dev.device] = true;
    return n;
}

template <bool A_MN, bool B_MN, int EPI>
tpmlp_status launch_splitk(const CUtensorMap& ma, const CUtensorMap& mb, const tc::KArgs& k, cudaStream_t st) {
    auto kern = tc::gemm_splitk_kernel<A_MN, B_MN, EPI>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4 * (k.num_tiles - k.tile_begin));  // one tile per cluster of four
    cfg.blockDim = dim3(tc::SK_THREADS);
    cfg.dynamicSmemBytes = tc::SK_SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 4;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddep_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, k);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("tcgen05 split-K GEMM launch: %s", cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    count_launch();
    return TPMLP_OK;
}

// Picks the tiling and launches.  CTA-pair 256x256 tiles when there are at least as many
// of them as co-resident pairs (or when forced); otherwise single-CTA 128x256 tiles, or
// 128x128 tiles when the 128x256 ones would leave more than half of the SMs idle.
// g.max_sms > 0 caps the grid at that many SMs (a GEMM run beside another on the rest).
// plan_out != nullptr: only report how the launch would run (GemmPlan), and launch nothing.
template <bool A_MN, bool B_MN, int EPI>
tpmlp_status launch_variant(const Operand& a, const Operand& b, const GemmSpec& g, tc::KArgs k, const DeviceInfo& dev,
                            cudaStream_t st, GemmPlan* plan_out = nullptr) {
    const int mode = g_gemm_mode.load(std::memory_order_relaxed);
    const int m_pairs = static_cast<int>((g.M + 2 * tc::BM - 1) / (2 * tc::BM));
    const int pair_tiles = m_pairs * k.n_blocks * k.batch;
    int cap = (mode == 1) ? 0 : pair_capacity<A_MN, B_MN, EPI, false>(dev);
    if (g.max_sms > 0 && cap > g.max_sms / 2) cap = g.max_sms / 2;
    const int sm_cap = g.max_sms > 0 && g.max_sms < dev.sm_count ? g.max_sms : dev.sm_count;
    bool use_pair = cap > 0 && ((mode >= 2 && mode <= 4) || pair_tiles >= cap);
    // Split-K CTA pairs for a shard-summing GEMM whose 256x256 tiles are fewer than the pairs the
    // GPU holds (it would otherwise run on single-CTA tiles), with a K loop long enough to split.
    constexpr bool kSplitOk = (EPI == EPI_BIAS_ACT && !A_MN && B_MN) || (EPI == EPI_STORE && !A_MN) ||
                              (EPI == EPI_STORE && A_MN && B_MN);
    bool split = false;
    int tail = 0;  // > 0: the last partial wave's tiles, run as split-K after the full waves
    if constexpr (kSplitOk) {
        if (g.sum_shards && !k.accumulate && k.k_iters >= 2 && cap > 0 &&
            (mode == 5 || (mode == 0 && pair_tiles < cap && k.k_iters >= 16)))
            split = splitk_capacity<A_MN, B_MN, EPI>(dev) >= pair_tiles && 4 * pair_tiles <= sm_cap;
        // A multi-wave GEMM whose last wave is at most half full: that wave's tiles on two CTA
        // pairs each with half the K loop (the pair kernel takes the full waves), so the wave
        // costs about half a tile time.
        const int rem = cap > 0 ? pair_tiles % cap : 0;
        // (long K loops only: their full waves keep the direct-store epilogue they would get anyway)
        if (!split && (mode == 0 || mode == 5) && !k.accumulate && g.max_sms == 0 && pair_tiles > cap && rem > 0 &&
            2 * rem <= cap && k.k_iters > kStagedMaxKBlocks && splitk_capacity<A_MN, B_MN, EPI>(dev) >= rem)
            tail = rem;
    }
    if (split) use_pair = true;  // pair-shaped operand boxes
    constexpr bool kNarrowOk = EPI != EPI_SWIGLU && EPI != EPI_DSWIGLU;  // packed layouts span 256 columns
    // Fewer pair tiles than pairs: single-CTA 128x256 tiles would occupy no more SMs (a pair tile is
    // two of them stacked) but move twice the B bytes per SM and store from registers, so the pairs
    // stay, unless 128x128 single-CTA tiles would occupy up to twice as many SMs.
    if (!use_pair && cap > 0 && (mode == 0 || mode == 5) && !(kNarrowOk && 2 * k.num_tiles <= dev.sm_count && g.N > 128))
        use_pair = true;
    const bool narrow = kNarrowOk && !use_pair && 2 * k.num_tiles <= dev.sm_count && g.N > 128;
    if (plan_out) {
        if (split) {
            *plan_out = GemmPlan{4 * pair_tiles, pair_tiles, pair_tiles, (k.k_iters + 1) / 2, 1, 0};
        } else if (use_pair) {
            const int clusters = pair_tiles < cap ? pair_tiles : cap;
            *plan_out = GemmPlan{2 * clusters, pair_tiles, clusters, k.k_iters, 0, tail};
        } else {
            const int tiles = narrow ? k.m_blocks * static_cast<int>((g.N + 127) / 128) * k.batch : k.num_tiles;
            const int grid = tiles < sm_cap ? tiles : sm_cap;
            *plan_out = GemmPlan{grid, tiles, grid, k.k_iters, 0, 0};
        }
        return TPMLP_OK;
    }
    CUtensorMap ma, mb;
    const uint32_t b_rows = (use_pair || narrow) ? tc::BN / 2 : tc::BN;
    // MN-major operands: one 4-D box per stage when the MN extent is a multiple of 64
    k.a_chunked = (a.mn_major && g.M % 64 == 0) ? 1 : 0;
    k.b_chunked = (b.mn_major && g.N % 64 == 0) ? 1 : 0;
    const uint32_t a_rows = tc::BM;
    bool ok;
    if (k.a_chunked) ok = make_map_chunked(&ma, a, g.M, g.K, tc::BM / 64);
    else ok = a.mn_major ? make_map(&ma, a, g.M, g.K, 64, tc::BK) : make_map(&ma, a, g.K, g.M, tc::BK, a_rows);
    if (!ok) return TPMLP_ERR_CUDA;
    if (k.b_chunked) ok = make_map_chunked(&mb, b, g.N, g.K, b_rows / 64);
    else ok = b.mn_major ? make_map(&mb, b, g.N, g.K, 64, tc::BK) : make_map(&mb, b, g.K, g.N, tc::BK, b_rows);
    if (!ok) return TPMLP_ERR_CUDA;
    if (!use_pair) {
        if constexpr (kNarrowOk) {
            if (narrow) {
                k.n_blocks = static_cast<int>((g.N + 127) / 128);
                k.num_tiles = k.m_blocks * k.n_blocks * k.batch;
                return launch_single<A_MN, B_MN, EPI, 128>(ma, mb, k, dev, sm_cap, st);
            }
        }
        return launch_single<A_MN, B_MN, EPI, 256>(ma, mb, k, dev, sm_cap, st);
    }
    k.m_blocks = m_pairs;
    k.num_tiles = pair_tiles;
    {
        // K reversal pays only across many waves of tiles (L2 reuse from one wave to the next);
        // a GEMM of at most two waves on the full grid walks K forwards on every grid, so its bits
        // do not depend on the grid.
        const int full = pair_capacity<A_MN, B_MN, EPI, false>(dev);  // the uncapped grid's clusters
        k.rev_period = (full > 0 && pair_tiles > 2 * full) ? full : INT_MAX;
    }
    if constexpr (kSplitOk) {
        if (split) return launch_splitk<A_MN, B_MN, EPI>(ma, mb, k, st);
        if (tail > 0) {
            tc::KArgs kf = k;  // the full waves on CTA pairs, direct-store epilogue (long K loops)
            kf.num_tiles = pair_tiles - tail;
            const tpmlp_status r = launch_pair<A_MN, B_MN, EPI, false>(ma, mb, ma, ma, kf, cap, st);
            if (r != TPMLP_OK) return r;
            if (g.tail_event != nullptr) {
                const cudaError_t e = cudaEventRecord(g.tail_event, st);
                if (e != cudaSuccess) {
                    set_error("event between a GEMM's full waves and its last wave: %s", cudaGetErrorString(e));
                    return TPMLP_ERR_CUDA;
                }
            }
            k.tile_begin = pair_tiles - tail;
            return launch_splitk<A_MN, B_MN, EPI>(ma, mb, k, st);
        }
    }
    const int clusters = pair_tiles < cap ? pair_tiles : cap;
    // Short K loops (a tile's main loop shorter than a direct-store epilogue): staged epilogue.
    if constexpr (kNarrowOk) {
        // (TMA stores overwrite: a launch that adds to its output stores directly)
        const bool staged = !k.accumulate && (mode == 4 || (mode != 3 && k.k_iters <= kStagedMaxKBlocks));
        if (staged && pair_capacity<A_MN, B_MN, EPI, true>(dev) >= clusters) {
            CUtensorMap mo, mo2 = ma;
            const uint64_t oshards = static_cast<uint64_t>(k.batch);
            if (!make_out_map(&mo, g.out, g.out_ld, g.out_ss, g.N, g.M, oshards, g.out_f32)) return TPMLP_ERR_CUDA;
            if (g.out2 != nullptr && !make_out_map(&mo2, g.out2, g.out2_ld, g.out2_ss, g.N, g.M, oshards, false))
                return TPMLP_ERR_CUDA;
            return launch_pair<A_MN, B_MN, EPI, true>(ma, mb, mo, mo2, k, clusters, st);
        }
    }
    return launch_pair<A_MN, B_MN, EPI, false>(ma, mb, ma, ma, k, clusters, st);
}

tpmlp_status launch_one(const Operand& a, const Operand& b, const GemmSpec& g, const DeviceInfo& dev,
                        cudaStream_t st, bool accumulate, GemmPlan* plan_out = nullptr) {
    tc::KArgs k{};
    k.accumulate = accumulate ? 1 : 0;
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
    k.group_m = g_group_m.load(std::memory_order_relaxed);
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
    {
        // 32-byte epilogue accesses need every row of out, out2 and aux to start on a 32-byte
        // boundary: base address, row pitch and shard stride all multiples of 32 bytes (the
        // column offsets inside a row are multiples of 32 elements).
        const int64_t shards = g.sum_shards ? 1 : g.n_shards;
        auto rows32 = [shards](const void* ptr, int64_t ld, int64_t ss, int64_t es) {
            if (ptr == nullptr) return true;
            return reinterpret_cast<uintptr_t>(ptr) % 32 == 0 && (ld * es) % 32 == 0 &&
                   (shards <= 1 || (ss * es) % 32 == 0);
        };
        const int64_t es_out = g.out_f32 ? 4 : 2;
        const int64_t es_out2 = g.epi == EPI_SWIGLU ? 4 : 2;  // fp32 SwiGLU pre-activations, else bf16 H
        const int64_t es_aux = g.epi == EPI_DSWIGLU ? 4 : 2;
        k.st32 = rows32(g.out, g.out_ld, g.out_ss, es_out) && rows32(g.out2, g.out2_ld, g.out2_ss, es_out2) &&
                         rows32(g.aux, g.aux_ld, g.aux_ss, es_aux)
                     ? 1
                     : 0;
    }
    if (k.num_tiles == 0) {
        if (plan_out) *plan_out = GemmPlan{0, 0, 0, 0, 0, 0};
        return TPMLP_OK;
    }

    const bool amn = a.mn_major, bmn = b.mn_major;
    if (g.epi == EPI_BIAS_ACT && !amn && bmn)
        return launch_variant<false, true, EPI_BIAS_ACT>(a, b, g, k, dev, st, plan_out);
    if (g.epi == EPI_DGELU && !amn && !bmn) return launch_variant<false, false, EPI_DGELU>(a, b, g, k, dev, st, plan_out);
    if (g.epi == EPI_SWIGLU && !amn && bmn) return launch_variant<false, true, EPI_SWIGLU>(a, b, g, k, dev, st, plan_out);
    if (g.epi == EPI_DSWIGLU && !amn && !bmn)
        return launch_variant<false, false, EPI_DSWIGLU>(a, b, g, k, dev, st, plan_out);
    if (g.epi == EPI_STORE && amn && bmn) return launch_variant<true, true, EPI_STORE>(a, b, g, k, dev, st, plan_out);
    if (g.epi == EPI_STORE && !amn && bmn) return launch_variant<false, true, EPI_STORE>(a, b, g, k, dev, st, plan_out);
    if (g.epi == EPI_STORE && !amn && !bmn)
        return launch_variant<false, false, EPI_STORE>(a, b, g, k, dev, st, plan_out);
    set_error("internal: no tcgen05 GEMM variant for epi=%d a_mn=%d b_mn=%d", g.epi, (int)amn, (int)bmn);
    return TPMLP_ERR_CUDA;
}

// The operand with its K origin moved to element k0 (K-major: a column offset; MN-major: a row
// offset).  bf16 operands only.
Operand shift_k(Operand o, int64_t k0) {
    o.ptr = static_cast<const char*>(o.ptr) + (o.mn_major ? k0 * o.ld : k0) * 2;
    return o;
}

}  // namespace

// The tensor cores' fp32 accumulation loses accuracy roughly in proportion to the number of
// 16-deep MMA steps it chains (measured: rel. Frobenius error 1.5e-4 at 2^13 steps, 2.5e-3 at
// 2^17), so an fp32-output contraction longer than the K chunk (default 4096 blocks of 64:
// the weight gradients of more than 262144 tokens) runs as one launch per K chunk: the first
// stores, each later one adds its partial product to the output in its epilogue (in fp32,
// rounded to nearest).  Each launch waits for the previous one's writes (griddepcontrol.wait
// before any global access), and the chunk order is fixed, so results stay deterministic.
tpmlp_status launch_tc_gemm(const Operand& a, const Operand& b, const GemmSpec& g, const DeviceInfo& dev,
                            cudaStream_t st) {
    const int64_t chunk = static_cast<int64_t>(g_k_chunk_blocks.load(std::memory_order_relaxed)) * tc::BK;
    if (g.epi != EPI_STORE || !g.out_f32 || g.sum_shards || g.K <= chunk)
        return launch_one(a, b, g, dev, st, false);
    for (int64_t k0 = 0; k0 < g.K; k0 += chunk) {
        GemmSpec gc = g;
        gc.K = g.K - k0 < chunk ? g.K - k0 : chunk;
        const tpmlp_status r = launch_one(shift_k(a, k0), shift_k(b, k0), gc, dev, st, k0 > 0);
        if (r != TPMLP_OK) return r;
    }
    return TPMLP_OK;
}

bool tc_gemm_plan(const Operand& a, const Operand& b, const GemmSpec& g, const DeviceInfo& dev, GemmPlan* plan) {
    // the first launch of a split contraction is the widest (each later one covers the same tiles)
    const int64_t chunk = static_cast<int64_t>(g_k_chunk_blocks.load(std::memory_order_relaxed)) * tc::BK;
    GemmSpec gc = g;
    if (g.epi == EPI_STORE && g.out_f32 && !g.sum_shards && g.K > chunk) gc.K = chunk;
    return launch_one(a, b, gc, dev, nullptr, false, plan) == TPMLP_OK;
}

int tc_gemm_sms(const Operand& a, const Operand& b, const GemmSpec& g, const DeviceInfo& dev) {
    GemmPlan pl{};
    if (!tc_gemm_plan(a, b, g, dev, &pl)) return dev.sm_count;
    return pl.sms;
}

void set_k_chunk_blocks(int blocks) {
    g_k_chunk_blocks.store(blocks > 0 ? blocks : kDefaultKChunkBlocks, std::memory_order_relaxed);
}
int get_k_chunk_blocks() { return g_k_chunk_blocks.load(std::memory_order_relaxed); }

void set_gemm_mode(int mode) { g_gemm_mode.store(mode, std::memory_order_relaxed); }
void set_group_m(int g) { g_group_m.store(g, std::memory_order_relaxed); }
int get_group_m() { return g_group_m.load(std::memory_order_relaxed); }
int get_gemm_mode() { return g_gemm_mode.load(std::memory_order_relaxed); }

}  // namespace tpmlp

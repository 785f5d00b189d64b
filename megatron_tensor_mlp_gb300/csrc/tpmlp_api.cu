// C-ABI front end: argument validation (host only, before any CUDA call),
// per-device state, and the mapping of each entry point onto GEMM launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace tpmlp {

// Device status word: written by kernels whose bounded waits give up.
__device__ uint32_t g_status_word;

namespace {
thread_local char t_err[512] = "";
std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ok[kMaxDevices];
std::mutex g_dev_mu;

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

int esize(tpmlp_dtype dt) { return dt == TPMLP_F32 ? 4 : 2; }

struct Range {
    const void* p;
    int64_t bytes;
};

bool overlap(const Range& a, const Range& b) {
    if (!a.p || !b.p || a.bytes <= 0 || b.bytes <= 0) return false;
    auto a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + static_cast<uintptr_t>(b.bytes) && b0 < a0 + static_cast<uintptr_t>(a.bytes);
}

// Outputs must not overlap inputs or each other.
tpmlp_status check_alias(std::initializer_list<Range> outs, std::initializer_list<Range> ins) {
    int i = 0;
    for (const Range& o : outs) {
        for (const Range& in : ins)
            if (overlap(o, in)) {
                set_error("output %d overlaps an input", i);
                return TPMLP_ERR_ALIAS;
            }
        int j = 0;
        for (const Range& o2 : outs) {
            if (j > i && overlap(o, o2)) {
                set_error("outputs %d and %d overlap", i, j);
                return TPMLP_ERR_ALIAS;
            }
            ++j;
        }
        ++i;
    }
    return TPMLP_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

tpmlp_status check_aligned(std::initializer_list<const void*> ptrs) {
    int i = 0;
    for (const void* p : ptrs) {
        if (p && !aligned16(p)) {
            set_error("pointer argument %d is not 16-byte aligned", i);
            return TPMLP_ERR_ALIGNMENT;
        }
        ++i;
    }
    return TPMLP_OK;
}

tpmlp_status check_pitch(int64_t elems, tpmlp_dtype dt, const char* what) {
    if ((elems * esize(dt)) % 16 != 0) {
        set_error("%s = %lld elements is not a multiple of 16 bytes", what, (long long)elems);
        return TPMLP_ERR_ALIGNMENT;
    }
    return TPMLP_OK;
}

// Common shape checks of the MLP entry points.
tpmlp_status check_mlp_shape(int64_t s, int64_t b, int64_t h, int64_t ffn, int p, bool need_h_div) {
    if (s < 0 || b < 0 || h < 1 || ffn < 1 || p < 1) {
        set_error("bad shape: s=%lld b=%lld h=%lld ffn=%lld p=%d", (long long)s, (long long)b, (long long)h,
                  (long long)ffn, p);
        return TPMLP_ERR_SHAPE;
    }
    if (h > kMaxDim || ffn > kMaxDim || (b > 0 && s > kMaxDim / b)) {
        set_error("shape too large: s*b, h and ffn must each be below 2^31");
        return TPMLP_ERR_SHAPE;
    }
    // every tensor of the block (with the 2x SwiGLU and 4-byte gradient widths) below 2^40 bytes
    const int64_t M = s * b, kMaxElems = (int64_t(1) << 40) / 16;
    if ((M > 0 && ffn > kMaxElems / M) || (M > 0 && h > kMaxElems / M) || ffn > kMaxElems / h) {
        set_error("shape too large: a tensor of the block would exceed 2^40 bytes");
        return TPMLP_ERR_SHAPE;
    }
    if (ffn % p != 0) {
        set_error("ffn=%lld is not divisible by p=%d", (long long)ffn, p);
        return TPMLP_ERR_DIVISIBILITY;
    }
    if (need_h_div && h % p != 0) {
        set_error("h=%lld is not divisible by p=%d", (long long)h, p);
        return TPMLP_ERR_DIVISIBILITY;
    }
    return TPMLP_OK;
}

tpmlp_status check_dtype(tpmlp_dtype dt) {
    if (dt != TPMLP_BF16 && dt != TPMLP_F32) {
        set_error("unknown dtype %d", (int)dt);
        return TPMLP_ERR_DTYPE;
    }
    return TPMLP_OK;
}

#define TP_TRY(expr)                          \
    do {                                      \
        tpmlp_status _st = (expr);            \
        if (_st != TPMLP_OK) return _st;      \
    } while (0)

tpmlp_status get_device(const DeviceInfo** out) {
    const DeviceInfo* d = device_info();
    if (!d) return TPMLP_ERR_CUDA;
    if (d->cc_major != 10 || d->cc_minor != 3) {
        set_error("device %d has compute capability %d.%d; this library is built for sm_103a (10.3) only", d->device,
                  d->cc_major, d->cc_minor);
        return TPMLP_ERR_ARCH;
    }
    *out = d;
    return TPMLP_OK;
}

tpmlp_status run_gemm(const Operand& a, const Operand& b, const GemmSpec& g, tpmlp_dtype dt, const DeviceInfo& dev,
                      cudaStream_t st) {
    if (dt == TPMLP_BF16) return launch_tc_gemm(a, b, g, dev, st);
    return launch_simt_gemm(a, b, g, dev, st);
}

GemmSpec spec_base() {
    GemmSpec g;
    std::memset(&g, 0, sizeof(g));
    return g;
}

// One GEMM launch: its operands and everything else.
struct GemmCall {
    Operand a, b;
    GemmSpec g;
};
tpmlp_status run_call(const GemmCall& c, tpmlp_dtype dt, const DeviceInfo& dev, cudaStream_t st, int max_sms = 0) {
    GemmSpec g = c.g;
    g.max_sms = max_sms;
    return run_gemm(c.a, c.b, g, dt, dev, st);
}

// Column layer: H_i = X A_i + b1_i, Y_i = act(H_i).  One launch over all p shards.
GemmCall column_call(const void* X, const void* A_sh, const void* b1_sh, void* Y_sh, void* H_sh, int64_t M,
                     int64_t h, int64_t ffn, int p, int act) {
    const int64_t fs = ffn / p;
    GemmCall c{{X, h, 0, 1, false},             // X [M][h], K-major
               {A_sh, fs, h * fs, p, true},     // A_i [h][fs]: [K][N], MN-major
               spec_base()};
    c.g.M = M; c.g.N = fs; c.g.K = h; c.g.n_shards = p;
    c.g.sum_shards = false; c.g.a_batched = false; c.g.b_batched = true;
    c.g.epi = EPI_BIAS_ACT; c.g.act = act;
    c.g.out = Y_sh; c.g.out_ld = fs; c.g.out_ss = M * fs;
    c.g.out2 = H_sh; c.g.out2_ld = fs; c.g.out2_ss = M * fs;
    c.g.bias = b1_sh; c.g.bias_ss = fs;
    return c;
}
tpmlp_status do_column(const void* X, const void* A_sh, const void* b1_sh, void* Y_sh, void* H_sh, int64_t M,
                       int64_t h, int64_t ffn, int p, tpmlp_dtype dt, int act, const DeviceInfo& dev,
                       cudaStream_t st) {
    return run_call(column_call(X, A_sh, b1_sh, Y_sh, H_sh, M, h, ffn, p, act), dt, dev, st);
}

// Row layer with the shard sum in the K loop: Z = sum_i Y_i B_i + b2.
GemmCall row_call(const void* Y_sh, const void* B_sh, const void* b2, void* Z, int64_t M, int64_t h, int64_t ffn,
                  int p) {
    const int64_t fs = ffn / p;
    GemmCall c{{Y_sh, fs, M * fs, p, false},    // Y_i [M][fs], K-major
               {B_sh, h, fs * h, p, true},      // B_i [fs][h]: [K][N], MN-major
               spec_base()};
    c.g.M = M; c.g.N = h; c.g.K = fs; c.g.n_shards = p;
    c.g.sum_shards = true;
    c.g.epi = EPI_BIAS_ACT; c.g.act = TPMLP_ACT_NONE;
    c.g.out = Z; c.g.out_ld = h; c.g.out_ss = 0;
    c.g.bias = b2; c.g.bias_ss = 0;
    return c;
}
tpmlp_status do_row(const void* Y_sh, const void* B_sh, const void* b2, void* Z, int64_t M, int64_t h, int64_t ffn,
                    int p, tpmlp_dtype dt, const DeviceInfo& dev, cudaStream_t st) {
    return run_call(row_call(Y_sh, B_sh, b2, Z, M, h, ffn, p), dt, dev, st);
}

// Row layer without the bias, its shard sum left in fp32: Z_part = sum_i Y_i B_i over the shards
// given (a rank's partial of a block whose shards are spread over several GPUs).
GemmCall row_partial_call(const void* Y_sh, const void* B_sh, float* Z_part, int64_t M, int64_t h, int64_t ffn,
                          int p) {
    GemmCall c = row_call(Y_sh, B_sh, nullptr, Z_part, M, h, ffn, p);
    c.g.epi = EPI_STORE; c.g.act = 0; c.g.out_f32 = true;
    return c;
}

// The block forward: the column GEMM, then the row GEMM.
tpmlp_status block_fwd(const GemmCall& col, const GemmCall& row, tpmlp_dtype dt, const DeviceInfo& dev,
                       cudaStream_t st) {
    TP_TRY(run_call(col, dt, dev, st));
    return run_call(row, dt, dev, st);
}

// dY_i = dZ B_i^T, times GeLU'(H_i) when act is GeLU (K = h)
GemmCall dY_call(const void* B_sh, const void* dZ, const void* H_sh, void* dY_sh, int64_t M, int64_t h, int64_t ffn,
                 int p, tpmlp_dtype dt, int act) {
    const int64_t fs = ffn / p;
    GemmCall c{{dZ, h, 0, 1, false},            // dZ [M][h]: [M][K]
               {B_sh, h, fs * h, p, false},     // B_i [fs][h]: [N][K], K-major
               spec_base()};
    c.g.M = M; c.g.N = fs; c.g.K = h; c.g.n_shards = p;
    c.g.a_batched = false; c.g.b_batched = true;
    if (act == TPMLP_ACT_GELU_ERF) {
        c.g.epi = EPI_DGELU;
        c.g.aux = H_sh; c.g.aux_ld = fs; c.g.aux_ss = M * fs;
    } else {
        c.g.epi = EPI_STORE;
        c.g.out_f32 = (dt == TPMLP_F32);
    }
    c.g.out = dY_sh; c.g.out_ld = fs; c.g.out_ss = M * fs;
    return c;
}
// dB_i = Y_i^T dZ (K = tokens)
GemmCall dB_call(const void* Y_sh, const void* dZ, void* dB_sh, int64_t M, int64_t h, int64_t ffn, int p,
                 bool grad_f32) {
    const int64_t fs = ffn / p;
    GemmCall c{{Y_sh, fs, M * fs, p, true},     // Y_i [M][fs]: [K][M_gemm], MN-major
               {dZ, h, 0, 1, true},             // dZ [M][h]: [K][N], MN-major
               spec_base()};
    c.g.M = fs; c.g.N = h; c.g.K = M; c.g.n_shards = p;
    c.g.a_batched = true; c.g.b_batched = false;
    c.g.epi = EPI_STORE; c.g.out_f32 = grad_f32;
    c.g.out = dB_sh; c.g.out_ld = h; c.g.out_ss = fs * h;
    return c;
}

// Row layer backward: dY_i = dZ B_i^T (times GeLU'(H_i) when act is GeLU), dB_i = Y_i^T dZ, db2.
tpmlp_status do_row_bwd(const void* Y_sh, const void* B_sh, const void* dZ, const void* H_sh, void* dY_sh,
                        void* dB_sh, void* db2, int64_t M, int64_t h, int64_t ffn, int p, tpmlp_dtype dt,
                        bool grad_f32, int act, const DeviceInfo& dev, cudaStream_t st) {
    TP_TRY(run_call(dY_call(B_sh, dZ, H_sh, dY_sh, M, h, ffn, p, dt, act), dt, dev, st));
    if (db2) TP_TRY(launch_colsum(dZ, dt == TPMLP_F32, 1, M, h, db2, grad_f32, st));
    return run_call(dB_call(Y_sh, dZ, dB_sh, M, h, ffn, p, grad_f32), dt, dev, st);
}

// Column sums run beside a GEMM on the caller's side stream (tpmlp_set_side_stream).
struct SideSums {
    const void* dZ; void* db2; const void* dH; void* db1; int64_t M, h, fs, p; bool f32;
    cudaStream_t side; cudaEvent_t fork, join;
};
tpmlp_status side_fork(const SideSums& w, cudaStream_t st);

// dA_i = X^T dY_i (K = tokens)
GemmCall dA_call(const void* X, const void* dY_sh, void* dA_sh, int64_t M, int64_t h, int64_t ffn, int p,
                 bool grad_f32) {
    const int64_t fs = ffn / p;
    GemmCall c{{X, h, 0, 1, true},              // X [M][h]: [K][M_gemm], MN-major
               {dY_sh, fs, M * fs, p, true},    // dY_i [M][fs]: [K][N], MN-major
               spec_base()};
    c.g.M = h; c.g.N = fs; c.g.K = M; c.g.n_shards = p;
    c.g.a_batched = false; c.g.b_batched = true;
    c.g.epi = EPI_STORE; c.g.out_f32 = grad_f32;
    c.g.out = dA_sh; c.g.out_ld = fs; c.g.out_ss = h * fs;
    return c;
}
// dX = sum_i dY_i A_i^T (the shard sum in the K loop); dX_f32: fp32 output
GemmCall dX_call(const void* dY_sh, const void* A_sh, void* dX, int64_t M, int64_t h, int64_t ffn, int p, bool dX_f32) {
    const int64_t fs = ffn / p;
    GemmCall c{{dY_sh, fs, M * fs, p, false},   // dY_i [M][fs], K-major
               {A_sh, fs, h * fs, p, false},    // A_i [h][fs]: [N][K], K-major
               spec_base()};
    c.g.M = M; c.g.N = h; c.g.K = fs; c.g.n_shards = p;
    c.g.sum_shards = true;
    c.g.epi = EPI_STORE; c.g.out_f32 = dX_f32;
    c.g.out = dX; c.g.out_ld = h; c.g.out_ss = 0;
    return c;
}

enum ForkAt { kForkNone = 0, kForkBeforeDA = 1, kForkBeforeDX = 2 };

// Column layer backward: dA_i = X^T dY_i, db1_i = 1^T dY_i, dX = sum_i dY_i A_i^T.
// dX_f32: dX is stored in fp32 (a rank's partial sum for an All-Reduce), else in dt.
// side / fork_at: the block's column sums to fork onto the side stream before the dA or dX launch.
tpmlp_status do_column_bwd(const void* X, const void* A_sh, const void* dY_sh, void* dX, void* dA_sh, void* db1_sh,
                           int64_t M, int64_t h, int64_t ffn, int p, tpmlp_dtype dt, bool grad_f32,
                           const DeviceInfo& dev, cudaStream_t st, bool dX_f32 = false,
                           const SideSums* side = nullptr, ForkAt fork_at = kForkNone) {
    const int64_t fs = ffn / p;
    if (db1_sh) TP_TRY(launch_colsum(dY_sh, dt == TPMLP_F32, p, M, fs, db1_sh, grad_f32, st));
    if (side && fork_at == kForkBeforeDA) TP_TRY(side_fork(*side, st));
    const GemmCall ca = dA_call(X, dY_sh, dA_sh, M, h, ffn, p, grad_f32);
    TP_TRY(run_gemm(ca.a, ca.b, ca.g, dt, dev, st));
    if (side && fork_at == kForkBeforeDX) TP_TRY(side_fork(*side, st));
    const GemmCall cx = dX_call(dY_sh, A_sh, dX, M, h, ffn, p, dX_f32 || dt == TPMLP_F32);
    return run_gemm(cx.a, cx.b, cx.g, dt, dev, st);
}

// A side stream and two events of the caller's (tpmlp_set_side_stream), per host thread.  The
// library never creates, destroys or synchronises them.
struct SideHandles {
    int device = -1;
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
thread_local SideHandles t_side;

tpmlp_status side_fork(const SideSums& w, cudaStream_t st) {
    cudaError_t e = cudaEventRecord(w.fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(w.side, w.fork, 0);
    if (e != cudaSuccess) {
        set_error("side stream fork: %s", cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    if (w.db2) TP_TRY(launch_colsum_any_sm(w.dZ, 1, w.M, w.h, w.db2, w.f32, w.side));
    if (w.db1) TP_TRY(launch_colsum_any_sm(w.dH, w.p, w.M, w.fs, w.db1, w.f32, w.side));
    e = cudaEventRecord(w.join, w.side);
    if (e != cudaSuccess) {
        set_error("side stream join: %s", cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    return TPMLP_OK;
}

// The column layer backward of a block (do_column_bwd) with the block's bias-gradient column sums,
// db1 of dY_sh and db2 of dZ (either may be NULL).  They run in line on `st`, or, when the caller
// has registered a side stream, on that stream beside the first of the dA and dX GEMMs whose
// persistent grid leaves enough SMs idle for all the sums' CTAs at once (one CTA per 256-column
// strip and shard): forked just before that GEMM's launch (an event recorded on `st`) and joined
// before anything that follows dX on `st`.  The GEMM's CTAs are resident by the time the fork
// event completes (programmatic launch), so the sums run only on the SMs it leaves idle.  A GEMM
// that fills every SM gets no sums beside it: they would take SMs its CTAs wait for (measured at
// the fwd+bwd bench workload, whose dX fills all 76 CTA pairs: backward 3-5 % slower).  Both
// ways give the same bits.
tpmlp_status column_bwd_with_db2(const void* X, const void* A_sh, const void* dY_sh, void* dX, void* dA_sh,
                                 void* db1_sh, const void* dZ, void* db2, int64_t M, int64_t h, int64_t ffn, int p,
                                 tpmlp_dtype dt, bool grad_f32, const DeviceInfo& dev, cudaStream_t st,
                                 bool dX_f32 = false) {
    const int64_t fs = ffn / p;
    ForkAt at = kForkNone;
    if (t_side.s != nullptr && t_side.device == dev.device && dt == TPMLP_BF16 && (db1_sh || db2)) {
        const int64_t strips = (db1_sh ? p * ((fs + 255) / 256) : 0) + (db2 ? (h + 255) / 256 : 0);
        const GemmCall ca = dA_call(X, dY_sh, dA_sh, M, h, ffn, p, grad_f32);
        const GemmCall cx = dX_call(dY_sh, A_sh, dX, M, h, ffn, p, dX_f32);
        if (dev.sm_count - tc_gemm_sms(ca.a, ca.b, ca.g, dev) >= strips) at = kForkBeforeDA;
        else if (dev.sm_count - tc_gemm_sms(cx.a, cx.b, cx.g, dev) >= strips) at = kForkBeforeDX;
    }
    if (at == kForkNone) {
        if (db2) TP_TRY(launch_colsum(dZ, dt == TPMLP_F32, 1, M, h, db2, grad_f32, st));
        return do_column_bwd(X, A_sh, dY_sh, dX, dA_sh, db1_sh, M, h, ffn, p, dt, grad_f32, dev, st, dX_f32);
    }
    const SideSums w{dZ, db2, dY_sh, db1_sh, M, h, fs, p, grad_f32, t_side.s, t_side.fork, t_side.join};
    TP_TRY(do_column_bwd(X, A_sh, dY_sh, dX, dA_sh, nullptr, M, h, ffn, p, dt, grad_f32, dev, st, dX_f32, &w, at));
    const cudaError_t e = cudaStreamWaitEvent(st, t_side.join, 0);
    if (e != cudaSuccess) {
        set_error("side stream join: %s", cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    return TPMLP_OK;
}

// ---------------------------------------------------------------- two GEMMs side by side
// A GEMM of one or two waves of tiles spends much of its launch filling its pipeline and
// draining its last tile's epilogue, with SMs idle behind its last partial wave.  Two
// independent ones -- dH_i and dB_i of the row layer's backward, dA_i and dX of the column
// layer's -- then finish sooner side by side, each on its share of the SMs, than one after the
// other.  Costs are in K-block times (one 64-deep K step of a CTA pair's 256x256 tile, about
// 0.27 us at the boost clock): a GEMM's waves of tiles, each the longer of its K loop and a
// short-K tile's epilogue, plus the last tile's epilogue, which nothing overlaps, plus the
// exchange of a split-K GEMM's partial sums.
constexpr double kEpilogueBlocks = 18.0;  // a short-K tile's epilogue (measured 4.5-5.7 us)
constexpr double kExchangeBlocks = 8.0;   // split-K partial sums through distributed shared memory (~2 us)
constexpr double kLaunchBlocks = 10.0;    // the gap between two dependent launches (~2.5-3 us)

// Cost of a GEMM on at most `sms` SMs (above), and in *used the SMs its grid occupies.
double gemm_cost(const GemmCall& c, const DeviceInfo& dev, int sms, int* used = nullptr) {
    GemmSpec g = c.g;
    g.max_sms = sms;
    GemmPlan pl{};
    if (used) *used = 0;
    if (!tc_gemm_plan(c.a, c.b, g, dev, &pl)) return 1e30;
    if (used) *used = pl.sms;
    if (pl.tiles == 0) return 0.0;
    if (pl.slots <= 0) return 1e30;
    const int waves = (pl.tiles + pl.slots - 1) / pl.slots;
    const double per_tile = pl.k_blocks > kEpilogueBlocks ? pl.k_blocks : kEpilogueBlocks;
    return waves * per_tile + kEpilogueBlocks + (pl.split_k ? kExchangeBlocks : 0.0);
}

// SMs for `a` when `a` and `b` should run side by side, or 0 when one after the other is about
// as fast.  Each candidate caps one GEMM's grid (even counts: CTA pairs take two) and gives the
// other every SM the first does not occupy; among equally fast splits the one leaving fewest
// SMs idle wins.
int side_by_side_sms(const GemmCall& a, const GemmCall& b, const DeviceInfo& dev) {
    const int S = dev.sm_count;
    const double apart = gemm_cost(a, dev, S) + gemm_cost(b, dev, S) + kLaunchBlocks;
    double best = apart;
    int best_x = 0, best_idle = S;
    auto consider = [&](double cost, int a_sms, int idle) {
        if (cost < best || (cost == best && best_x > 0 && idle < best_idle)) {
            best = cost;
            best_x = a_sms;
            best_idle = idle;
        }
    };
    for (int x = 2; x + 2 <= S; x += 2) {
        int ua = 0, ub = 0;
        const double ca = gemm_cost(a, dev, x, &ua);  // a capped at x, b on the rest
        const double cb = gemm_cost(b, dev, S - ua, &ub);
        if (ua > 0 && ub > 0) consider(std::max(ca, cb), ua, S - ua - ub);
        const double cb2 = gemm_cost(b, dev, x, &ub);  // b capped at x, a on the rest
        const double ca2 = gemm_cost(a, dev, S - ub, &ua);
        if (ua > 0 && ub > 0) consider(std::max(ca2, cb2), S - ub, S - ua - ub);
    }
    return best < 0.9 * apart ? best_x : 0;  // the fork and join cost a little too
}

// The two splits of a backward (dH | dB, dA | dX), remembered per shape for this thread.
struct SplitKey {
    int64_t M, h, ffn;
    int p, device, mode, group_m, gf32, dx32;
    bool operator==(const SplitKey& o) const {
        return M == o.M && h == o.h && ffn == o.ffn && p == o.p && device == o.device && mode == o.mode &&
               group_m == o.group_m && gf32 == o.gf32 && dx32 == o.dx32;
    }
};
struct SplitMemo {
    SplitKey key[4];
    int x1[4], x2[4];
    int n = 0, next = 0;
};
thread_local SplitMemo t_split;

void backward_splits(const GemmCall& dy, const GemmCall& db, const GemmCall& da, const GemmCall& dx, const SplitKey& key,
                     const DeviceInfo& dev, int* x1, int* x2) {
    for (int i = 0; i < t_split.n; ++i) {
        if (t_split.key[i] == key) {
            *x1 = t_split.x1[i];
            *x2 = t_split.x2[i];
            return;
        }
    }
    *x1 = side_by_side_sms(dy, db, dev);
    *x2 = side_by_side_sms(da, dx, dev);
    const int i = t_split.next;
    t_split.key[i] = key;
    t_split.x1[i] = *x1;
    t_split.x2[i] = *x2;
    t_split.next = (i + 1) % 4;
    if (t_split.n < 4) ++t_split.n;
}

tpmlp_status record_and_wait(cudaEvent_t ev, cudaStream_t from, cudaStream_t to, const char* what) {
    cudaError_t e = cudaEventRecord(ev, from);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(to, ev, 0);
    if (e != cudaSuccess) {
        set_error("%s: %s", what, cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    return TPMLP_OK;
}

// A block backward's column sums beside the last waves of its weight-gradient GEMMs (the GeLU
// block's dB_i and dA_i; the SwiGLU block's dB_i and packed dW_i).  A GEMM
// of several waves whose last wave is at most half full runs that wave as a second, short
// launch on four CTAs per tile (split-K CTA pairs), which leaves most SMs idle while it runs
// (at s=2048 b=4 h=5120 ffn=20480 p=4: dB_i and dA_i, 4 tiles on 16 of 152 SMs for ~25 us).
// When dB_i's or dA_i's last wave leaves at least half the SMs idle, the side stream waits for
// an event recorded between that GEMM's two launches (GemmSpec::tail_event) and sums there --
// db2 beside dB_i's last wave, db1 beside dA_i's (both beside the one there is) -- and `st`
// waits for the sums before its next GEMM, whose persistent grid then finds every SM free: the
// sums cost the time by which they outlast the last wave, instead of their whole time in line.
// The same column-sum kernel runs either way, so the bits do not change.  *done = false when
// neither GEMM has such a last wave (nothing launched: the caller runs the backward in line).
struct SumsBesideTails {
    const void* dZ; void* db2; const void* dH; void* db1; int64_t M, h, fs, p; bool f32;
};
tpmlp_status sums_beside_tails(const GemmCall& dy, const GemmCall& db, const GemmCall& da, const GemmCall& dx,
                               const SumsBesideTails& w, tpmlp_dtype dt, const DeviceInfo& dev, cudaStream_t st,
                               bool* done) {
    *done = false;
    auto roomy_tail = [&](const GemmCall& c) {
        GemmPlan pl{};
        return tc_gemm_plan(c.a, c.b, c.g, dev, &pl) && pl.tail > 0 && 2 * (4 * pl.tail) <= dev.sm_count;
    };
    const bool at_db = roomy_tail(db), at_da = roomy_tail(da);
    if (!at_db && !at_da) return TPMLP_OK;
    *done = true;
    cudaStream_t ss = t_side.s;
    auto db2_sum = [&](cudaStream_t on) { return launch_colsum(w.dZ, false, 1, w.M, w.h, w.db2, w.f32, on); };
    auto db1_sum = [&](cudaStream_t on) { return launch_colsum(w.dH, false, w.p, w.M, w.fs, w.db1, w.f32, on); };
    // GEMM c on st with the sums marked `mine` beside its last wave.  The fork event is recorded
    // once before the GEMM and again between its two launches; should the launch run no separate
    // last wave after all, the sums still start after everything before the GEMM (correct, only
    // not beside the last wave).
    auto gemm_with_sums = [&](const GemmCall& c, bool mine2, bool mine1) -> tpmlp_status {
        const bool fork = (mine2 && w.db2) || (mine1 && w.db1);
        if (!fork) return run_call(c, dt, dev, st);
        cudaError_t e = cudaEventRecord(t_side.fork, st);
        if (e != cudaSuccess) {
            set_error("side stream fork: %s", cudaGetErrorString(e));
            return TPMLP_ERR_CUDA;
        }
        GemmCall cc = c;
        cc.g.tail_event = t_side.fork;
        TP_TRY(run_call(cc, dt, dev, st));
        e = cudaStreamWaitEvent(ss, t_side.fork, 0);
        if (e != cudaSuccess) {
            set_error("side stream fork: %s", cudaGetErrorString(e));
            return TPMLP_ERR_CUDA;
        }
        if (mine2 && w.db2) TP_TRY(db2_sum(ss));
        if (mine1 && w.db1) TP_TRY(db1_sum(ss));
        return record_and_wait(t_side.join, ss, st, "side stream join");
    };
    // every sum is assigned to exactly one of the two GEMMs
    TP_TRY(run_call(dy, dt, dev, st));
    TP_TRY(gemm_with_sums(db, at_db, at_db && !at_da));
    TP_TRY(gemm_with_sums(da, !at_db, at_da));
    return run_call(dx, dt, dev, st);
}

// The block backward (GeLU' fused) from dZ.  With a side stream of the caller's registered
// (tpmlp_set_side_stream) and a split that pays (side_by_side_sms), the two pairs of independent
// GEMMs run side by side:
//   st:   dH_i (x1 SMs)            | db1, dA_i = X^T dH_i (x2 SMs)
//   side: dB_i (the rest), db2     | dX = sum_i dH_i A_i^T (the rest)
// The side stream starts after everything before it on `st`, starts dX only after dH, and `st`
// waits for it before returning; a phase whose split does not pay runs both its GEMMs on `st`.
// Every tile keeps its accumulation order on a smaller grid, so dH, dB, dA and the column sums
// have the same bits either way; dX may run on CTA pairs rather than split-K pairs in a
// narrower share, which adds its fp32 partial sums in another order.  Otherwise: do_row_bwd
// and column_bwd_with_db2.  dX_f32: dX is a rank's fp32 partial sum.
tpmlp_status block_bwd(const void* X, const void* A_sh, const void* B_sh, const void* H_sh, const void* Y_sh,
                       const void* dZ, void* dX, void* dA_sh, void* dB_sh, void* db1_sh, void* db2, void* dH_ws,
                       int64_t M, int64_t h, int64_t ffn, int p, tpmlp_dtype dt, bool gf32, bool dX_f32,
                       const DeviceInfo& dev, cudaStream_t st) {
    int x1 = 0, x2 = 0;
    const bool side = t_side.s != nullptr && t_side.device == dev.device && dt == TPMLP_BF16;
    const GemmCall dy = dY_call(B_sh, dZ, H_sh, dH_ws, M, h, ffn, p, dt, TPMLP_ACT_GELU_ERF);
    const GemmCall db = dB_call(Y_sh, dZ, dB_sh, M, h, ffn, p, gf32);
    const GemmCall da = dA_call(X, dH_ws, dA_sh, M, h, ffn, p, gf32);
    const GemmCall dx = dX_call(dH_ws, A_sh, dX, M, h, ffn, p, dX_f32 || dt == TPMLP_F32);
    if (side) {
        const SplitKey key{M, h, ffn, p, dev.device, get_gemm_mode(), get_group_m(), gf32 ? 1 : 0, dX_f32 ? 1 : 0};
        backward_splits(dy, db, da, dx, key, dev, &x1, &x2);
    }
    if (x1 == 0 && x2 == 0) {
        if (side && (db1_sh || db2)) {
            const int64_t fs = ffn / p;
            const SumsBesideTails w{dZ, db2, dH_ws, db1_sh, M, h, fs, p, gf32};
            bool done = false;
            TP_TRY(sums_beside_tails(dy, db, da, dx, w, dt, dev, st, &done));
            if (done) return TPMLP_OK;
        }
        TP_TRY(do_row_bwd(Y_sh, B_sh, dZ, H_sh, dH_ws, dB_sh, nullptr, M, h, ffn, p, dt, gf32, TPMLP_ACT_GELU_ERF,
                          dev, st));
        return column_bwd_with_db2(X, A_sh, dH_ws, dX, dA_sh, db1_sh, dZ, db2, M, h, ffn, p, dt, gf32, dev, st,
                                   dX_f32);
    }
    const int S = dev.sm_count;
    const int64_t fs = ffn / p;
    cudaStream_t ss = t_side.s;
    TP_TRY(record_and_wait(t_side.fork, st, ss, "side stream fork"));
    if (x1 > 0) {
        TP_TRY(run_call(db, dt, dev, ss, S - x1));
        if (db2) TP_TRY(launch_colsum(dZ, false, 1, M, h, db2, gf32, ss));
        TP_TRY(run_call(dy, dt, dev, st, x1));
    } else {
        TP_TRY(run_call(dy, dt, dev, st));
        if (db2) TP_TRY(launch_colsum(dZ, false, 1, M, h, db2, gf32, st));
        TP_TRY(run_call(db, dt, dev, st));
    }
    if (x2 > 0) {
        TP_TRY(record_and_wait(t_side.fork, st, ss, "side stream fork"));  // dH is complete
        TP_TRY(run_call(dx, dt, dev, ss, S - x2));
        if (db1_sh) TP_TRY(launch_colsum(dH_ws, false, p, M, fs, db1_sh, gf32, st));
        TP_TRY(run_call(da, dt, dev, st, x2));
    } else {
        if (db1_sh) TP_TRY(launch_colsum(dH_ws, false, p, M, fs, db1_sh, gf32, st));
        TP_TRY(run_call(da, dt, dev, st));
        TP_TRY(run_call(dx, dt, dev, st));
    }
    return record_and_wait(t_side.join, ss, st, "side stream join");
}

// SwiGLU shape rules: ffn/p a multiple of 128 (gate/up blocks of 128 features), bf16 only.
tpmlp_status check_swiglu(int64_t ffn, int p, tpmlp_dtype dt) {
    if (dt != TPMLP_BF16) {
        set_error("the SwiGLU block runs on bf16 tensors only");
        return TPMLP_ERR_DTYPE;
    }
    if ((ffn / p) % 128 != 0) {
        set_error("SwiGLU needs ffn/p to be a multiple of 128 (ffn=%lld, p=%d)", (long long)ffn, p);
        return TPMLP_ERR_DIVISIBILITY;
    }
    return TPMLP_OK;
}

}  // namespace

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(t_err, sizeof(t_err), fmt, ap);
    va_end(ap);
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

const DeviceInfo* device_info() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error("cudaGetDevice: %s", cudaGetErrorString(e));
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        set_error("device index %d out of range", dev);
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev_ok[dev]) {
        DeviceInfo d{};
        d.device = dev;
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) {
            set_error("cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
            return nullptr;
        }
        if (d.cc_major == 10 && d.cc_minor == 3) {
            void* addr = nullptr;
            if ((e = cudaGetSymbolAddress(&addr, g_status_word)) != cudaSuccess) {
                set_error("cudaGetSymbolAddress(status word): %s", cudaGetErrorString(e));
                return nullptr;
            }
            d.status = static_cast<uint32_t*>(addr);
        }
        g_dev[dev] = d;
        g_dev_ok[dev] = true;
    }
    return &g_dev[dev];
}

}  // namespace tpmlp

using namespace tpmlp;

extern "C" {

tpmlp_status tpmlp_column_fwd(const void* X, const void* A_sh, const void* b1_sh, void* Y_sh, void* H_sh, int64_t s,
                              int64_t b, int64_t h, int64_t ffn, int p, tpmlp_dtype dt, tpmlp_act act, void* stream) {
    if (!X || !A_sh || !Y_sh) {
        set_error("X, A_sh and Y_sh must not be NULL");
        return TPMLP_ERR_NULL;
    }
    TP_TRY(check_mlp_shape(s, b, h, ffn, p, false));
    TP_TRY(check_dtype(dt));
    if (act != TPMLP_ACT_NONE && act != TPMLP_ACT_GELU_ERF) {
        set_error("unknown activation %d", (int)act);
        return TPMLP_ERR_DTYPE;
    }
    const int64_t M = s * b, fs = ffn / p, es = esize(dt);
    TP_TRY(check_aligned({X, A_sh, b1_sh, Y_sh, H_sh}));
    TP_TRY(check_pitch(h, dt, "h"));
    TP_TRY(check_pitch(fs, dt, "ffn/p"));
    TP_TRY(check_alias({{Y_sh, M * ffn * es}, {H_sh, M * ffn * es}},
                       {{X, M * h * es}, {A_sh, h * ffn * es}, {b1_sh, ffn * es}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (M == 0) return TPMLP_OK;
    return do_column(X, A_sh, b1_sh, Y_sh, H_sh, M, h, ffn, p, dt, act, *dev, static_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_row_fwd(const void* Y_sh, const void* B_sh, const void* b2, void* Z, int64_t s, int64_t b,
                           int64_t h, int64_t ffn, int p, tpmlp_dtype dt, void* stream) {
    if (!Y_sh || !B_sh || !Z) {
        set_error("Y_sh, B_sh and Z must not be NULL");
        return TPMLP_ERR_NULL;
    }
    TP_TRY(check_mlp_shape(s, b, h, ffn, p, false));
    TP_TRY(check_dtype(dt));
    const int64_t M = s * b, fs = ffn / p, es = esize(dt);
    TP_TRY(check_aligned({Y_sh, B_sh, b2, Z}));
    TP_TRY(check_pitch(h, dt, "h"));
    TP_TRY(check_pitch(fs, dt, "ffn/p"));
    TP_TRY(check_alias({{Z, M * h * es}}, {{Y_sh, M * ffn * es}, {B_sh, ffn * h * es}, {b2, h * es}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (M == 0) return TPMLP_OK;
    return do_row(Y_sh, B_sh, b2, Z, M, h, ffn, p, dt, *dev, static_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_mlp_fwd(const void* X, const void* A_sh, const void* b1_sh, const void* B_sh, const void* b2,
                           void* Z, void* Y_ws, void* H_sh, int64_t s, int64_t b, int64_t h, int64_t ffn, int p,
                           tpmlp_dtype dt, void* stream) {
    if (!X || !A_sh || !B_sh || !Z || !Y_ws) {
        set_error("X, A_sh, B_sh, Z and Y_ws must not be NULL");
        return TPMLP_ERR_NULL;
    }
    TP_TRY(check_mlp_shape(s, b, h, ffn, p, true));
    TP_TRY(check_dtype(dt));
    const int64_t M = s * b, fs = ffn / p, es = esize(dt);
    TP_TRY(check_aligned({X, A_sh, b1_sh, B_sh, b2, Z, Y_ws, H_sh}));
    TP_TRY(check_pitch(h, dt, "h"));
    TP_TRY(check_pitch(fs, dt, "ffn/p"));
    TP_TRY(check_alias({{Z, M * h * es}, {Y_ws, M * ffn * es}, {H_sh, M * ffn * es}},
                       {{X, M * h * es}, {A_sh, h * ffn * es}, {b1_sh, ffn * es}, {B_sh, ffn * h * es},
                        {b2, h * es}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (M == 0) return TPMLP_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return block_fwd(column_call(X, A_sh, b1_sh, Y_ws, H_sh, M, h, ffn, p, TPMLP_ACT_GELU_ERF),
                     row_call(Y_ws, B_sh, b2, Z, M, h, ffn, p), dt, *dev, st);
}

tpmlp_status tpmlp_mlp_bwd(const void* X, const void* A_sh, const void* B_sh, const void* H_sh, const void* Y_sh,
                           const void* dZ, void* dX, void* dA_sh, void* dB_sh, void* db1_sh, void* db2, void* dH_ws,
                           int64_t s, int64_t b, int64_t h, int64_t ffn, int p, tpmlp_dtype dt, tpmlp_dtype grad_dt,
                           void* stream) {
    if (!X || !A_sh || !B_sh || !H_sh || !Y_sh || !dZ || !dX || !dA_sh || !dB_sh || !dH_ws) {
        set_error("only db1_sh and db2 may be NULL");
        return TPMLP_ERR_NULL;
    }
    TP_TRY(check_mlp_shape(s, b, h, ffn, p, true));
    TP_TRY(check_dtype(dt));
    TP_TRY(check_dtype(grad_dt));
    if (dt == TPMLP_F32 && grad_dt != TPMLP_F32) {
        set_error("grad_dt must be TPMLP_F32 when dt is TPMLP_F32");
        return TPMLP_ERR_DTYPE;
    }
    const int64_t M = s * b, fs = ffn / p, es = esize(dt), gs = esize(grad_dt);
    TP_TRY(check_aligned({X, A_sh, B_sh, H_sh, Y_sh, dZ, dX, dA_sh, dB_sh, db1_sh, db2, dH_ws}));
    TP_TRY(check_pitch(h, dt, "h"));
    TP_TRY(check_pitch(fs, dt, "ffn/p"));
    TP_TRY(check_alias({{dX, M * h * es}, {dA_sh, h * ffn * gs}, {dB_sh, ffn * h * gs}, {db1_sh, ffn * gs},
                        {db2, h * gs}, {dH_ws, M * ffn * es}},
                       {{X, M * h * es}, {A_sh, h * ffn * es}, {B_sh, ffn * h * es}, {H_sh, M * ffn * es},
                        {Y_sh, M * ffn * es}, {dZ, M * h * es}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (M == 0) return TPMLP_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // row layer backward with GeLU' fused: dH_i = (dZ B_i^T) * GeLU'(H_i); dB_i; db2; then the
    // column layer backward from dH: db1_i, dA_i, dX = sum_i dH_i A_i^T
    return block_bwd(X, A_sh, B_sh, H_sh, Y_sh, dZ, dX, dA_sh, dB_sh, db1_sh, db2, dH_ws, M, h, ffn, p, dt,
                     grad_dt == TPMLP_F32, false, *dev, st);
}

tpmlp_status tpmlp_mlp_fwd_partial(const void* X, const void* A_sh, const void* b1_sh, const void* B_sh, float* Z_part,
                                   void* Y_ws, void* H_sh, int64_t s, int64_t b, int64_t h, int64_t ffn, int p,
                                   tpmlp_dtype dt, void* stream) {
    if (!X || !A_sh || !B_sh || !Z_part || !Y_ws) {
        set_error("X, A_sh, B_sh, Z_part and Y_ws must not be NULL");
        return TPMLP_ERR_NULL;
    }
    TP_TRY(check_mlp_shape(s, b, h, ffn, p, true));
    TP_TRY(check_dtype(dt));
    const int64_t M = s * b, fs = ffn / p, es = esize(dt);
    TP_TRY(check_aligned({X, A_sh, b1_sh, B_sh, Z_part, Y_ws, H_sh}));
    TP_TRY(check_pitch(h, dt, "h"));
    TP_TRY(check_pitch(fs, dt, "ffn/p"));
    TP_TRY(check_alias({{Z_part, M * h * 4}, {Y_ws, M * ffn * es}, {H_sh, M * ffn * es}},
                       {{X, M * h * es}, {A_sh, h * ffn * es}, {b1_sh, ffn * es}, {B_sh, ffn * h * es}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (M == 0) return TPMLP_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return block_fwd(column_call(X, A_sh, b1_sh, Y_ws, H_sh, M, h, ffn, p, TPMLP_ACT_GELU_ERF),
                     row_partial_call(Y_ws, B_sh, Z_part, M, h, ffn, p), dt, *dev, st);
}

tpmlp_status tpmlp_mlp_bwd_partial(const void* X, const void* A_sh, const void* B_sh, const void* H_sh,
                                   const void* Y_sh, const void* dZ, float* dX_part, void* dA_sh, void* dB_sh,
                                   void* db1_sh, void* db2, void* dH_ws, int64_t s, int64_t b, int64_t h,
                                   int64_t ffn, int p, tpmlp_dtype dt, tpmlp_dtype grad_dt, void* stream) {
    if (!X || !A_sh || !B_sh || !H_sh || !Y_sh || !dZ || !dX_part || !dA_sh || !dB_sh || !dH_ws) {
        set_error("only db1_sh and db2 may be NULL");
        return TPMLP_ERR_NULL;
    }
    TP_TRY(check_mlp_shape(s, b, h, ffn, p, true));
    TP_TRY(check_dtype(dt));
    TP_TRY(check_dtype(grad_dt));
    if (dt == TPMLP_F32 && grad_dt != TPMLP_F32) {
        set_error("grad_dt must be TPMLP_F32 when dt is TPMLP_F32");
        return TPMLP_ERR_DTYPE;
    }
    const int64_t M = s * b, fs = ffn / p, es = esize(dt), gs = esize(grad_dt);
    TP_TRY(check_aligned({X, A_sh, B_sh, H_sh, Y_sh, dZ, dX_part, dA_sh, dB_sh, db1_sh, db2, dH_ws}));
    TP_TRY(check_pitch(h, dt, "h"));
    TP_TRY(check_pitch(fs, dt, "ffn/p"));
    TP_TRY(check_alias({{dX_part, M * h * 4}, {dA_sh, h * ffn * gs}, {dB_sh, ffn * h * gs}, {db1_sh, ffn * gs},
                        {db2, h * gs}, {dH_ws, M * ffn * es}},
                       {{X, M * h * es}, {A_sh, h * ffn * es}, {B_sh, ffn * h * es}, {H_sh, M * ffn * es},
                        {Y_sh, M * ffn * es}, {dZ, M * h * es}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (M == 0) return TPMLP_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return block_bwd(X, A_sh, B_sh, H_sh, Y_sh, dZ, dX_part, dA_sh, dB_sh, db1_sh, db2, dH_ws, M, h, ffn, p, dt,
                     grad_dt == TPMLP_F32, /*dX_f32=*/true, *dev, st);
}

tpmlp_status tpmlp_sum_finish(const float* S, const void* bias, void* out, int64_t rows, int64_t cols, tpmlp_dtype dt,
                              void* stream) {
    if (!S || !out) {
        set_error("S and out must not be NULL");
        return TPMLP_ERR_NULL;
    }
    if (rows < 0 || cols < 1 || rows > kMaxDim || cols > kMaxDim || (rows > 0 && cols > ((int64_t(1) << 40) / 4) / rows)) {
        set_error("bad shape rows=%lld cols=%lld", (long long)rows, (long long)cols);
        return TPMLP_ERR_SHAPE;
    }
    TP_TRY(check_dtype(dt));
    TP_TRY(check_aligned({S, bias, out}));
    TP_TRY(check_pitch(cols, dt, "cols"));
    TP_TRY(check_alias({{out, rows * cols * esize(dt)}}, {{S, rows * cols * 4}, {bias, cols * esize(dt)}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (rows == 0) return TPMLP_OK;
    return launch_sum_finish(S, bias, out, rows, cols, dt == TPMLP_F32, dev->sm_count,
                             static_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_row_bwd(const void* Y_sh, const void* B_sh, const void* dZ, const void* H_sh, void* dY_sh,
                           void* dB_sh, void* db2, int64_t s, int64_t b, int64_t h, int64_t ffn, int p, tpmlp_dtype dt,
                           tpmlp_dtype grad_dt, tpmlp_act act, void* stream) {
    if (!Y_sh || !B_sh || !dZ || !dY_sh || !dB_sh || (act == TPMLP_ACT_GELU_ERF && !H_sh)) {
        set_error("Y_sh, B_sh, dZ, dY_sh, dB_sh (and H_sh when act is GeLU) must not be NULL");
        return TPMLP_ERR_NULL;
    }
    TP_TRY(check_mlp_shape(s, b, h, ffn, p, false));
    TP_TRY(check_dtype(dt));
    TP_TRY(check_dtype(grad_dt));
    if (act != TPMLP_ACT_NONE && act != TPMLP_ACT_GELU_ERF) {
        set_error("unknown activation %d", (int)act);
        return TPMLP_ERR_DTYPE;
    }
    if (dt == TPMLP_F32 && grad_dt != TPMLP_F32) {
        set_error("grad_dt must be TPMLP_F32 when dt is TPMLP_F32");
        return TPMLP_ERR_DTYPE;
    }
    const int64_t M = s * b, fs = ffn / p, es = esize(dt), gs = esize(grad_dt);
    TP_TRY(check_aligned({Y_sh, B_sh, dZ, H_sh, dY_sh, dB_sh, db2}));
    TP_TRY(check_pitch(h, dt, "h"));
    TP_TRY(check_pitch(fs, dt, "ffn/p"));
    TP_TRY(check_alias({{dY_sh, M * ffn * es}, {dB_sh, ffn * h * gs}, {db2, h * gs}},
                       {{Y_sh, M * ffn * es}, {B_sh, ffn * h * es}, {dZ, M * h * es},
                        {act == TPMLP_ACT_GELU_ERF ? H_sh : nullptr, M * ffn * es}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (M == 0) return TPMLP_OK;
    return do_row_bwd(Y_sh, B_sh, dZ, H_sh, dY_sh, dB_sh, db2, M, h, ffn, p, dt, grad_dt == TPMLP_F32, act, *dev,
                      static_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_column_bwd(const void* X, const void* A_sh, const void* dY_sh, void* dX, void* dA_sh, void* db1_sh,
                              int64_t s, int64_t b, int64_t h, int64_t ffn, int p, tpmlp_dtype dt, tpmlp_dtype grad_dt,
                              void* stream) {
    if (!X || !A_sh || !dY_sh || !dX || !dA_sh) {
        set_error("only db1_sh may be NULL");
        return TPMLP_ERR_NULL;
    }
    TP_TRY(check_mlp_shape(s, b, h, ffn, p, false));
    TP_TRY(check_dtype(dt));
    TP_TRY(check_dtype(grad_dt));
    if (dt == TPMLP_F32 && grad_dt != TPMLP_F32) {
        set_error("grad_dt must be TPMLP_F32 when dt is TPMLP_F32");
        return TPMLP_ERR_DTYPE;
    }
    const int64_t M = s * b, fs = ffn / p, es = esize(dt), gs = esize(grad_dt);
    TP_TRY(check_aligned({X, A_sh, dY_sh, dX, dA_sh, db1_sh}));
    TP_TRY(check_pitch(h, dt, "h"));
    TP_TRY(check_pitch(fs, dt, "ffn/p"));
    TP_TRY(check_alias({{dX, M * h * es}, {dA_sh, h * ffn * gs}, {db1_sh, ffn * gs}},
                       {{X, M * h * es}, {A_sh, h * ffn * es}, {dY_sh, M * ffn * es}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (M == 0) return TPMLP_OK;
    return do_column_bwd(X, A_sh, dY_sh, dX, dA_sh, db1_sh, M, h, ffn, p, dt, grad_dt == TPMLP_F32, *dev,
                         static_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_swiglu_mlp_fwd(const void* X, const void* W_sh, const void* bw_sh, const void* B_sh,
                                  const void* b2, void* Z, void* Y_ws, void* H_ws, int64_t s, int64_t b, int64_t h,
                                  int64_t ffn, int p, tpmlp_dtype dt, void* stream) {
    if (!X || !W_sh || !B_sh || !Z || !Y_ws) {
        set_error("X, W_sh, B_sh, Z and Y_ws must not be NULL");
        return TPMLP_ERR_NULL;
    }
    TP_TRY(check_mlp_shape(s, b, h, ffn, p, true));
    TP_TRY(check_dtype(dt));
    TP_TRY(check_swiglu(ffn, p, dt));
    const int64_t M = s * b, fs = ffn / p, es = esize(dt);
    TP_TRY(check_aligned({X, W_sh, bw_sh, B_sh, b2, Z, Y_ws, H_ws}));
    TP_TRY(check_pitch(h, dt, "h"));
    TP_TRY(check_alias({{Z, M * h * es}, {Y_ws, M * ffn * es}, {H_ws, 2 * M * ffn * 4}},
                       {{X, M * h * es}, {W_sh, 2 * h * ffn * es}, {bw_sh, 2 * ffn * es}, {B_sh, ffn * h * es},
                        {b2, h * es}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (M == 0) return TPMLP_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    {
        Operand a{X, h, 0, 1, false};                  // X [M][h], K-major
        Operand bb{W_sh, 2 * fs, h * 2 * fs, p, true};  // packed [gate|up] W_i [h][2 fs], MN-major
        GemmSpec g = spec_base();
        g.M = M; g.N = 2 * fs; g.K = h; g.n_shards = p;
        g.a_batched = false; g.b_batched = true;
        g.epi = EPI_SWIGLU;
        g.out = Y_ws; g.out_ld = fs; g.out_ss = M * fs;
        g.out2 = H_ws; g.out2_ld = 2 * fs; g.out2_ss = M * 2 * fs;
        g.bias = bw_sh; g.bias_ss = 2 * fs;
        TP_TRY(run_gemm(a, bb, g, dt, *dev, st));
    }
    return do_row(Y_ws, B_sh, b2, Z, M, h, ffn, p, dt, *dev, st);
}

tpmlp_status tpmlp_swiglu_mlp_bwd(const void* X, const void* W_sh, const void* B_sh, const void* H_ws,
                                  const void* Y_ws, const void* dZ, void* dX, void* dW_sh, void* dB_sh, void* dbw_sh,
                                  void* db2, void* dH_ws, int64_t s, int64_t b, int64_t h, int64_t ffn, int p,
                                  tpmlp_dtype dt, tpmlp_dtype grad_dt, void* stream) {
    if (!X || !W_sh || !B_sh || !H_ws || !Y_ws || !dZ || !dX || !dW_sh || !dB_sh || !dH_ws) {
        set_error("only dbw_sh and db2 may be NULL");
        return TPMLP_ERR_NULL;
    }
    TP_TRY(check_mlp_shape(s, b, h, ffn, p, true));
    TP_TRY(check_dtype(dt));
    TP_TRY(check_dtype(grad_dt));
    TP_TRY(check_swiglu(ffn, p, dt));
    const int64_t M = s * b, fs = ffn / p, es = esize(dt), gs = esize(grad_dt);
    TP_TRY(check_aligned({X, W_sh, B_sh, H_ws, Y_ws, dZ, dX, dW_sh, dB_sh, dbw_sh, db2, dH_ws}));
    TP_TRY(check_pitch(h, dt, "h"));
    TP_TRY(check_alias({{dX, M * h * es}, {dW_sh, 2 * h * ffn * gs}, {dB_sh, ffn * h * gs}, {dbw_sh, 2 * ffn * gs},
                        {db2, h * gs}, {dH_ws, 2 * M * ffn * es}},
                       {{X, M * h * es}, {W_sh, 2 * h * ffn * es}, {B_sh, ffn * h * es}, {H_ws, 2 * M * ffn * 4},
                        {Y_ws, M * ffn * es}, {dZ, M * h * es}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (M == 0) return TPMLP_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool gf32 = grad_dt == TPMLP_F32;
    // dY = dZ B_i^T per feature; the epilogue writes the packed (dHg, dHu)
    GemmCall dy{{dZ, h, 0, 1, false}, {B_sh, h, fs * h, p, false}, spec_base()};
    dy.g.M = M; dy.g.N = fs; dy.g.K = h; dy.g.n_shards = p;
    dy.g.a_batched = false; dy.g.b_batched = true;
    dy.g.epi = EPI_DSWIGLU;
    dy.g.aux = H_ws; dy.g.aux_ld = 2 * fs; dy.g.aux_ss = M * 2 * fs;
    dy.g.out = dH_ws; dy.g.out_ld = 2 * fs; dy.g.out_ss = M * 2 * fs;
    const GemmCall db = dB_call(Y_ws, dZ, dB_sh, M, h, ffn, p, gf32);  // dB_i = Y_i^T dZ
    // the packed gate/up layer is a column layer of width 2 ffn: dW = X^T dH, dX = sum_i dH_i W_i^T
    if (t_side.s != nullptr && t_side.device == dev->device && (dbw_sh || db2)) {
        const GemmCall dw = dA_call(X, dH_ws, dW_sh, M, h, 2 * ffn, p, gf32);
        const GemmCall dx = dX_call(dH_ws, W_sh, dX, M, h, 2 * ffn, p, false);
        const SumsBesideTails w{dZ, db2, dH_ws, dbw_sh, M, h, 2 * fs, p, gf32};
        bool done = false;
        TP_TRY(sums_beside_tails(dy, db, dw, dx, w, dt, *dev, st, &done));
        if (done) return TPMLP_OK;
    }
    TP_TRY(run_call(dy, dt, *dev, st));
    TP_TRY(run_call(db, dt, *dev, st));
    return column_bwd_with_db2(X, W_sh, dH_ws, dX, dW_sh, dbw_sh, dZ, db2, M, h, 2 * ffn, p, dt, gf32, *dev, st);
}

tpmlp_status tpmlp_swiglu_pack(void* G, void* U, void* W_sh, int64_t rows, int64_t ffn, int p, tpmlp_dtype dt,
                               int inverse, void* stream) {
    if (!G || !U || !W_sh) {
        set_error("pointers must not be NULL");
        return TPMLP_ERR_NULL;
    }
    if (rows < 0 || ffn < 1 || p < 1 || rows > kMaxDim || ffn > kMaxDim) {
        set_error("bad shape rows=%lld ffn=%lld p=%d", (long long)rows, (long long)ffn, p);
        return TPMLP_ERR_SHAPE;
    }
    if (rows > 0 && 2 * ffn > ((int64_t(1) << 40) / 4) / rows) {
        set_error("shape too large: the packed matrix would exceed 2^40 bytes");
        return TPMLP_ERR_SHAPE;
    }
    if (ffn % p != 0 || (ffn / p) % 128 != 0) {
        set_error("SwiGLU packing needs ffn %% p == 0 and ffn/p a multiple of 128");
        return TPMLP_ERR_DIVISIBILITY;
    }
    TP_TRY(check_dtype(dt));
    TP_TRY(check_aligned({G, U, W_sh}));
    const int64_t bytes = rows * ffn * esize(dt);
    if (!inverse) TP_TRY(check_alias({{W_sh, 2 * bytes}}, {{G, bytes}, {U, bytes}}));
    else TP_TRY(check_alias({{G, bytes}, {U, bytes}}, {{W_sh, 2 * bytes}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (rows == 0) return TPMLP_OK;
    return launch_swiglu_pack(G, U, W_sh, rows, ffn, p, esize(dt), inverse != 0, static_cast<cudaStream_t>(stream));
}

static tpmlp_status shard_common(const void* src, void* dst, int64_t rows, int64_t cols, int p, tpmlp_dtype dt,
                                 bool inverse, void* stream) {
    if (!src || !dst) {
        set_error("pointers must not be NULL");
        return TPMLP_ERR_NULL;
    }
    if (rows < 0 || cols < 1 || p < 1 || rows > kMaxDim || cols > kMaxDim) {
        set_error("bad shape rows=%lld cols=%lld p=%d", (long long)rows, (long long)cols, p);
        return TPMLP_ERR_SHAPE;
    }
    if (rows > 0 && cols > ((int64_t(1) << 40) / 4) / rows) {
        set_error("shape too large: the matrix would exceed 2^40 bytes");
        return TPMLP_ERR_SHAPE;
    }
    if (cols % p != 0) {
        set_error("cols=%lld is not divisible by p=%d", (long long)cols, p);
        return TPMLP_ERR_DIVISIBILITY;
    }
    TP_TRY(check_dtype(dt));
    TP_TRY(check_aligned({src, dst}));
    TP_TRY(check_pitch(cols / p, dt, "cols/p"));
    const int64_t bytes = rows * cols * esize(dt);
    TP_TRY(check_alias({{dst, bytes}}, {{src, bytes}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (rows == 0) return TPMLP_OK;
    return launch_shard_columns(src, dst, rows, cols, p, esize(dt), inverse, static_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_shard_columns(const void* W, void* W_sh, int64_t rows, int64_t cols, int p, tpmlp_dtype dt,
                                 void* stream) {
    return shard_common(W, W_sh, rows, cols, p, dt, false, stream);
}

tpmlp_status tpmlp_unshard_columns(const void* W_sh, void* W, int64_t rows, int64_t cols, int p, tpmlp_dtype dt,
                                   void* stream) {
    return shard_common(W_sh, W, rows, cols, p, dt, true, stream);
}

tpmlp_status tpmlp_qkv_interleave(const void* W_qkv, void* W_out, int64_t rows, int64_t h, int64_t n_heads, int p,
                                  tpmlp_dtype dt, int inverse, void* stream) {
    if (!W_qkv || !W_out) {
        set_error("pointers must not be NULL");
        return TPMLP_ERR_NULL;
    }
    if (rows < 0 || h < 1 || n_heads < 1 || p < 1 || rows > kMaxDim || h > kMaxDim / 3) {
        set_error("bad shape rows=%lld h=%lld n_heads=%lld p=%d", (long long)rows, (long long)h, (long long)n_heads, p);
        return TPMLP_ERR_SHAPE;
    }
    if (rows > 0 && 3 * h > ((int64_t(1) << 40) / 4) / rows) {
        set_error("shape too large: the matrix would exceed 2^40 bytes");
        return TPMLP_ERR_SHAPE;
    }
    if (h % n_heads != 0 || n_heads % p != 0) {
        set_error("need h %% n_heads == 0 and n_heads %% p == 0 (h=%lld n_heads=%lld p=%d)", (long long)h,
                  (long long)n_heads, p);
        return TPMLP_ERR_DIVISIBILITY;
    }
    TP_TRY(check_dtype(dt));
    TP_TRY(check_aligned({W_qkv, W_out}));
    const int64_t bytes = rows * 3 * h * esize(dt);
    TP_TRY(check_alias({{W_out, bytes}}, {{W_qkv, bytes}}));
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    if (rows == 0) return TPMLP_OK;
    return launch_qkv_interleave(W_qkv, W_out, rows, h, n_heads, esize(dt), inverse != 0,
                                 static_cast<cudaStream_t>(stream));
}

int64_t tpmlp_qkv_src_col(int64_t dst_col, int64_t h, int64_t n_heads) {
    if (h < 1 || n_heads < 1 || h % n_heads != 0 || dst_col < 0 || dst_col >= 3 * h) return -1;
    const int64_t d = h / n_heads;
    const int64_t blk = dst_col / d, e = dst_col % d;
    return (blk % 3) * h + (blk / 3) * d + e;
}

tpmlp_status tpmlp_device_status(void* stream) {
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        set_error("cudaStreamSynchronize: %s", cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    uint32_t v = 0;
    if ((e = cudaMemcpy(&v, dev->status, sizeof(v), cudaMemcpyDeviceToHost)) != cudaSuccess) {
        set_error("reading the status word: %s", cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    if (v == 0) return TPMLP_OK;
    const uint32_t zero = 0;
    if ((e = cudaMemcpy(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess) {
        set_error("clearing the status word: %s", cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    if (v & kStatusTimeout) {
        set_error("a device-side wait gave up (where=%u)", v & 0xFFFFu);
        return TPMLP_ERR_TIMEOUT;
    }
    set_error("device status word 0x%x", v);
    return TPMLP_ERR_DEVICE;
}

tpmlp_status tpmlp_debug_wait_timeout(uint32_t timeout_us, void* stream) {
    if (timeout_us < 1 || timeout_us > 1000000) {
        set_error("timeout_us must be in 1..1000000");
        return TPMLP_ERR_SHAPE;
    }
    const DeviceInfo* dev;
    TP_TRY(get_device(&dev));
    return launch_debug_wait(timeout_us, dev->status, static_cast<cudaStream_t>(stream));
}

const char* tpmlp_status_string(tpmlp_status st) {
    switch (st) {
    case TPMLP_OK: return "TPMLP_OK";
    case TPMLP_ERR_NULL: return "TPMLP_ERR_NULL";
    case TPMLP_ERR_SHAPE: return "TPMLP_ERR_SHAPE";
    case TPMLP_ERR_DIVISIBILITY: return "TPMLP_ERR_DIVISIBILITY";
    case TPMLP_ERR_DTYPE: return "TPMLP_ERR_DTYPE";
    case TPMLP_ERR_ALIGNMENT: return "TPMLP_ERR_ALIGNMENT";
    case TPMLP_ERR_ALIAS: return "TPMLP_ERR_ALIAS";
    case TPMLP_ERR_ARCH: return "TPMLP_ERR_ARCH";
    case TPMLP_ERR_CUDA: return "TPMLP_ERR_CUDA";
    case TPMLP_ERR_TIMEOUT: return "TPMLP_ERR_TIMEOUT";
    case TPMLP_ERR_DEVICE: return "TPMLP_ERR_DEVICE";
    }
    return "TPMLP_ERR_UNKNOWN";
}

const char* tpmlp_last_error(void) { return t_err; }

int tpmlp_version(void) { return 200; }

uint64_t tpmlp_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

tpmlp_status tpmlp_set_side_stream(void* side_stream, void* fork_event, void* join_event) {
    if (!side_stream && !fork_event && !join_event) {
        t_side = SideHandles{};
        return TPMLP_OK;
    }
    if (!side_stream || !fork_event || !join_event) {
        set_error("side_stream, fork_event and join_event must all be given, or all be NULL");
        return TPMLP_ERR_NULL;
    }
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error("cudaGetDevice: %s", cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    t_side.device = dev;
    t_side.s = static_cast<cudaStream_t>(side_stream);
    t_side.fork = static_cast<cudaEvent_t>(fork_event);
    t_side.join = static_cast<cudaEvent_t>(join_event);
    return TPMLP_OK;
}

tpmlp_status tpmlp_set_gemm_mode(int mode) {
    if (mode < 0 || mode > 5) {
        set_error("gemm mode must be 0 (automatic), 1 (single-CTA tiles), 2 (CTA-pair tiles), 3 (CTA-pair tiles, "
                  "direct stores), 4 (CTA-pair tiles, TMA stores) or 5 (automatic, split-K forced)");
        return TPMLP_ERR_SHAPE;
    }
    set_gemm_mode(mode);
    return TPMLP_OK;
}

int tpmlp_get_gemm_mode(void) { return get_gemm_mode(); }

tpmlp_status tpmlp_set_gemm_raster(int group_m) {
    if (group_m < 1 || group_m > 1024) {
        set_error("group_m must be in 1..1024");
        return TPMLP_ERR_SHAPE;
    }
    set_group_m(group_m);
    return TPMLP_OK;
}

int tpmlp_get_gemm_raster(void) { return get_group_m(); }

tpmlp_status tpmlp_set_k_chunk(int k_blocks) {
    if (k_blocks < 0 || k_blocks > (1 << 24)) {
        set_error("k_blocks must be 0 (default) or in 1..2^24");
        return TPMLP_ERR_SHAPE;
    }
    set_k_chunk_blocks(k_blocks);
    return TPMLP_OK;
}

int tpmlp_get_k_chunk(void) { return get_k_chunk_blocks(); }

}  // extern "C"

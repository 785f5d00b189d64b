// Internal interfaces between the C-ABI front end (tpmlp_api.cu) and the
// kernel translation units.  Not part of the public header.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/tpmlp.h"

namespace tpmlp {

// Epilogue kinds of the GEMM kernels.
enum EpiKind : int {
    EPI_BIAS_ACT = 0,  // out = act(acc + bias[n]); optional out2 = acc + bias (pre-activation)
    EPI_DGELU = 1,     // out = acc * GeLU'(aux[m][n])
    EPI_STORE = 2,     // out = acc (fp32 or bf16)
    EPI_SWIGLU = 3,    // packed [gate 128 | up 128] tiles: out = silu(g + bg) * (u + bu); out2 = packed fp32 pre-activations
    EPI_DSWIGLU = 4,   // acc = dY per feature; reads packed fp32 (g, u) from aux, writes packed bf16 (dg, du)
};

// One operand of D[M,N] = sum_k A[M,K] B[K,N], batched over shards.
//   Element (row r, col c) of a [rows, cols] row-major slice of shard s lives at
//   ptr + s * ss + r * ld + c  (element units).
//   For A: "K-major" means the slice is [M][K] (K contiguous), "MN-major" [K][M].
//   For B: "K-major" means the slice is [N][K], "MN-major" [K][N].
struct Operand {
    const void* ptr;
    int64_t ld;       // row pitch (elements)
    int64_t ss;       // shard stride (elements)
    int64_t shards;   // number of shards stored (1 = not sharded)
    bool mn_major;
};

// Everything the GEMM kernels need besides the two operands.
struct GemmSpec {
    int64_t M, N, K;     // per-shard GEMM sizes
    int64_t n_shards;    // batch count (batched) or K-chunk count (sum_shards)
    bool sum_shards;     // true: D = sum_s A_s B_s in one accumulator; false: D_s = A_s B_s
    bool a_batched, b_batched;  // batched mode: operand follows the tile's shard (else shard 0)
    int epi;             // EpiKind
    int act;             // tpmlp_act (EPI_BIAS_ACT)
    bool out_f32;        // output element type (bf16 otherwise)
    void* out; int64_t out_ld, out_ss;
    void* out2; int64_t out2_ld, out2_ss;         // pre-activation save (EPI_BIAS_ACT), may be null
    const void* bias; int64_t bias_ss;            // [shard][N] of the input dtype, may be null
    const void* aux; int64_t aux_ld, aux_ss;      // EPI_DGELU: H
    int max_sms;         // > 0: the launch occupies at most this many SMs (a GEMM run beside another)
    cudaEvent_t tail_event;  // non-null: recorded on the stream between the full waves and the split-K
                             // last wave, when the GEMM runs one (GemmPlan::tail > 0)
};

// How a tcgen05 GEMM would run (tc_gemm_plan): the SMs its grid occupies, its work tiles, how
// many of them are in flight at once, the K blocks (of 64) each CTA pair or CTA accumulates
// per tile, whether two CTA pairs split each tile's K loop, and how many tiles of a last
// partial wave run after the full waves as a second launch on split-K CTA pairs (four CTAs
// per tile).
struct GemmPlan {
    int sms;
    int tiles;
    int slots;
    int k_blocks;
    int split_k;
    int tail;
};

struct DeviceInfo {
    int device;
    int sm_count;
    int cc_major, cc_minor;
    uint32_t* status;  // device address of this device's status word
};

// Per-device cached properties; nullptr (with last error set) on failure.
const DeviceInfo* device_info();

void set_error(const char* fmt, ...);

// Adds one to the process-wide count of kernels this library has launched
// (tpmlp_launch_count); every launcher calls it once per accepted launch.
void count_launch();

// Kernel launchers (all return TPMLP_OK or TPMLP_ERR_CUDA with the message set).
tpmlp_status launch_tc_gemm(const Operand& a, const Operand& b, const GemmSpec& g, const DeviceInfo& dev,
                            cudaStream_t st);
tpmlp_status launch_simt_gemm(const Operand& a, const Operand& b, const GemmSpec& g, const DeviceInfo& dev,
                              cudaStream_t st);
// out[s][n] = sum_m in[s][m][n]; in bf16 or f32 (in_f32), out f32 or bf16 (out_f32)
tpmlp_status launch_colsum(const void* in, bool in_f32, int64_t shards, int64_t M, int64_t N, void* out,
                           bool out_f32, cudaStream_t st);
// bf16 column sums without clusters, bit-identical to launch_colsum's (any free SM can run them)
tpmlp_status launch_colsum_any_sm(const void* in, int64_t shards, int64_t M, int64_t N, void* out, bool out_f32,
                                  cudaStream_t st);
tpmlp_status launch_shard_columns(const void* src, void* dst, int64_t rows, int64_t cols, int p, int esize,
                                  bool inverse, cudaStream_t st);
tpmlp_status launch_qkv_interleave(const void* src, void* dst, int64_t rows, int64_t h, int64_t n_heads,
                                   int esize, bool inverse, cudaStream_t st);
tpmlp_status launch_debug_wait(uint32_t timeout_us, uint32_t* status, cudaStream_t st);
// out[r][c] = S[r][c] + bias[c] rounded to the output type (bf16, or fp32 when out_f32)
tpmlp_status launch_sum_finish(const float* S, const void* bias, void* out, int64_t rows, int64_t cols, bool out_f32,
                               int sm_count, cudaStream_t st);
// SwiGLU packed layout: W_sh[i][r][256 b + j] = (j < 128 ? G : U)[r][i fs + 128 b + j % 128]
tpmlp_status launch_swiglu_pack(void* G, void* U, void* W_sh, int64_t rows, int64_t ffn, int p, int esize,
                                bool inverse, cudaStream_t st);

// How a bf16 GEMM launch of launch_tc_gemm would run, by the same tiling decision (false when
// no tcgen05 variant takes it); nothing is launched.  A K-chunked fp32 contraction reports its
// first launch.
bool tc_gemm_plan(const Operand& a, const Operand& b, const GemmSpec& g, const DeviceInfo& dev, GemmPlan* plan);
// SMs such a launch occupies for its whole run (its persistent grid: CTA pairs or single CTAs,
// one per SM).
int tc_gemm_sms(const Operand& a, const Operand& b, const GemmSpec& g, const DeviceInfo& dev);
// Process-wide GEMM tiling mode (see tpmlp_set_gemm_mode).
void set_gemm_mode(int mode);
int get_gemm_mode();
void set_group_m(int g);
int get_group_m();
// K blocks (of 64) per launch of a split fp32-output contraction (see launch_tc_gemm); <= 0 restores the default.
void set_k_chunk_blocks(int blocks);
int get_k_chunk_blocks();


}  // namespace tpmlp

// The MLP block forward for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) where they run this
// block: a plugin inside an inference engine that owns all device memory and
// offers no allocation during execution, or a runtime that fixes its memory
// budget at start-up and forbids allocation afterwards (an allocation can
// synchronise the device and break its latency guarantees).  tpmlp_mlp_fwd
// needs a caller-provided workspace for the intermediate activation Y; this
// entry point keeps Y in a fixed array inside the library instead, so such a
// caller passes only inputs and the output.
//
// The array is a file-scope __device__ object of TPMLP_NOALLOC_SCRATCH_BYTES:
// every GPU that loads the library holds it until the process exits.  Host
// code cannot hand the array's name to a kernel (on the host that name is only
// a stand-in, not a device address), so the first call on each device looks
// up the device address with cudaGetSymbolAddress, with that device current,
// and caches it.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace tpmlp {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[TPMLP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
void* g_scratch_addr[kMaxDev];
bool g_scratch_ready[kMaxDev];
std::mutex g_scratch_mu;

// Device address of this device's scratch array (set up once per device).
tpmlp_status scratch_address(const DeviceInfo& dev, void** out) {
    if (dev.device < 0 || dev.device >= kMaxDev) {
        set_error("device index %d out of range", dev.device);
        return TPMLP_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ready[dev.device]) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            set_error("cudaGetSymbolAddress(no-allocation scratch): %s", cudaGetErrorString(e));
            return TPMLP_ERR_CUDA;
        }
        g_scratch_addr[dev.device] = ptr;
        g_scratch_ready[dev.device] = true;
    }
    *out = g_scratch_addr[dev.device];
    return TPMLP_OK;
}

}  // namespace
}  // namespace tpmlp

using namespace tpmlp;

extern "C" tpmlp_status tpmlp_mlp_fwd_noalloc(const void* X, const void* A_sh, const void* b1_sh, const void* B_sh,
                                              const void* b2, void* Z, int64_t s, int64_t b, int64_t h,
                                              int64_t ffn, int p, tpmlp_dtype dt, void* stream) {
    if (!X || !A_sh || !B_sh || !Z) {
        set_error("X, A_sh, B_sh and Z must not be NULL");
        return TPMLP_ERR_NULL;
    }
    if (s < 0 || b < 0 || h < 1 || ffn < 1 || p < 1 || (b > 0 && s > ((int64_t(1) << 31) - 1) / b)) {
        set_error("bad shape: s=%lld b=%lld h=%lld ffn=%lld p=%d", (long long)s, (long long)b, (long long)h,
                  (long long)ffn, p);
        return TPMLP_ERR_SHAPE;
    }
    if (ffn % p != 0 || h % p != 0) {
        set_error("h=%lld and ffn=%lld must be divisible by p=%d", (long long)h, (long long)ffn, p);
        return TPMLP_ERR_DIVISIBILITY;
    }
    if (dt != TPMLP_BF16 && dt != TPMLP_F32) {
        set_error("unknown dtype %d", (int)dt);
        return TPMLP_ERR_DTYPE;
    }
    const int64_t M = s * b, es = dt == TPMLP_F32 ? 4 : 2;
    const int64_t cap = static_cast<int64_t>(TPMLP_NOALLOC_SCRATCH_BYTES);
    if (M > 0 && ffn > cap / (es * M)) {
        set_error("the intermediate activation needs s*b*ffn*%lld = %lld*%lld*%lld bytes; the no-allocation "
                  "entry point holds at most %lld bytes (use tpmlp_mlp_fwd with a caller workspace)",
                  (long long)es, (long long)M, (long long)ffn, (long long)es, (long long)cap);
        return TPMLP_ERR_SHAPE;
    }
    const DeviceInfo* dev = device_info();
    if (!dev) return TPMLP_ERR_CUDA;
    if (dev->cc_major != 10 || dev->cc_minor != 3) {
        set_error("device %d has compute capability %d.%d; this library is built for sm_103a (10.3) only",
                  dev->device, dev->cc_major, dev->cc_minor);
        return TPMLP_ERR_ARCH;
    }
    if (M == 0) return TPMLP_OK;
    void* Y = nullptr;
    tpmlp_status st = scratch_address(*dev, &Y);
    if (st != TPMLP_OK) return st;
    // The column layer writes every element of Y before the row layer reads it,
    // so nothing left in the array by an earlier call is ever read.
    st = tpmlp_column_fwd(X, A_sh, b1_sh, Y, nullptr, s, b, h, ffn, p, dt, TPMLP_ACT_GELU_ERF, stream);
    if (st != TPMLP_OK) return st;
    return tpmlp_row_fwd(Y, B_sh, b2, Z, s, b, h, ffn, p, dt, stream);
}

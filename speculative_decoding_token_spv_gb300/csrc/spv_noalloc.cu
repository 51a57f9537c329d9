// spv_noalloc.cu -- spv_verify_chain for callers that cannot allocate device
// memory.
//
// Some callers have no way to hand this library a workspace: a serving loop
// whose device memory is entirely pre-reserved by its own pool, a host
// program that links this library but manages no device memory, or code
// running where cudaMalloc is not permitted (inside a stream capture) or
// would stall the device at the wrong moment (cudaMalloc/cudaFree may
// synchronise).  spv_verify_chain_noalloc serves them: it runs the same
// kernels as spv_verify_chain, with the scratch space taken from a
// fixed-size array that lives in the library's own device memory.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds SPV_NOALLOC_SCRATCH_BYTES of device memory for it until the
// process exits.  Host code cannot use the array's name as a device address;
// the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and keeps it.
#include "spv.h"
#include "spv_internal.h"

#include <atomic>
#include <cmath>
#include <cstdint>

namespace {

static __device__ __align__(256) unsigned char spv_noalloc_scratch[SPV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_ptr[kMaxDevices];

// Device address of this device's copy of the scratch array (set up once per
// device, on the first call made with that device current).
cudaError_t scratch_address(int dev, void **out)
{
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        cudaError_t e = cudaGetSymbolAddress(&p, spv_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" spv_status spv_verify_chain_noalloc(const void *target_logits, const void *draft_logits,
                                               spv_dtype dtype, const int32_t *draft_tokens, const float *r,
                                               const uint64_t *sample_keys, int B, int gamma, int V,
                                               float temperature, int32_t *accept_count, int32_t *out_tokens,
                                               float *out_pq, float *out_resid_norm, int32_t *row_status,
                                               void *stream)
{
    if ((dtype != SPV_F32 && dtype != SPV_BF16) || !target_logits || !draft_tokens || !accept_count ||
        !out_tokens)
        return SPV_ERR_INVALID_ARG;
    if (gamma < 1 || gamma > SPV_MAX_GAMMA || B < 1 || V < 2) return SPV_ERR_INVALID_ARG;
    if (static_cast<double>(B) * (2 * gamma + 1) * V >= 9.0e15) return SPV_ERR_INVALID_ARG;
    if (!(temperature >= 0.0f) || std::isinf(temperature)) return SPV_ERR_INVALID_ARG;
    const bool greedy = temperature == 0.0f;
    if (!greedy && (!draft_logits || !r || !sample_keys)) return SPV_ERR_INVALID_ARG;
    if (!greedy && !(1.0f / temperature < INFINITY)) return SPV_ERR_INVALID_ARG;
    const size_t need = greedy ? spv::greedy_ws_bytes(B, gamma, V) : spv::chain_ws_bytes(B, gamma, V);
    if (need > static_cast<size_t>(SPV_NOALLOC_SCRATCH_BYTES)) return SPV_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPV_ERR_CUDA;
    void *scratch = nullptr;
    if (scratch_address(dev, &scratch) != cudaSuccess) return SPV_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The first word of the scratch is the timeout flag: start each call clear.
    if (cudaMemsetAsync(scratch, 0, sizeof(unsigned), st) != cudaSuccess) return SPV_ERR_CUDA;

    spv::ChainLaunch L{};
    L.target = target_logits;
    L.draft = draft_logits;
    L.dtype = dtype == SPV_F32 ? 0 : 1;
    L.tokens = draft_tokens;
    L.r = r;
    L.keys = sample_keys;
    L.B = B;
    L.gamma = gamma;
    L.V = V;
    L.T = temperature;
    L.accept_count = accept_count;
    L.out_tokens = out_tokens;
    L.out_pq = out_pq;
    L.out_Z = out_resid_norm;
    L.row_status = row_status;
    L.ws = scratch;
    const int eb = dtype == SPV_F32 ? 4 : 2;
    L.tma = (static_cast<size_t>(V) * eb) % 16 == 0 && aligned16(target_logits) && (greedy || aligned16(draft_logits));
    const cudaError_t e = greedy ? spv::launch_greedy(L, st) : spv::launch_chain(L, st);
    return e == cudaSuccess ? SPV_OK : SPV_ERR_CUDA;
}

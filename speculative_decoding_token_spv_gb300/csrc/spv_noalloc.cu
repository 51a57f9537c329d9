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
#include <cstdint>

namespace {

static __device__ __align__(256) unsigned char spv_noalloc_scratch[SPV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
constexpr size_t kHeaderClearBytes = 16;  // error word, self-test flag, work-item counter
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

}  // namespace

extern "C" spv_status spv_verify_chain_noalloc(const void *target_logits, const void *draft_logits,
                                               spv_dtype dtype, const int32_t *draft_tokens, const float *r,
                                               const uint64_t *sample_keys, int B, int gamma, int V,
                                               float temperature, int32_t *accept_count, int32_t *out_tokens,
                                               float *out_pq, float *out_resid_norm, int32_t *row_status,
                                               void *stream)
{
    const spv::ChainArgs a{target_logits, draft_logits, dtype, draft_tokens, r, sample_keys, B, gamma, V,
                           temperature, accept_count, out_tokens, out_pq, out_resid_norm, row_status};
    const spv_status chk = spv::check_chain_args(a);
    if (chk != SPV_OK) return chk;
    if (spv::chain_call_ws_bytes(a) > static_cast<size_t>(SPV_NOALLOC_SCRATCH_BYTES)) return SPV_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPV_ERR_CUDA;
    void *scratch = nullptr;
    if (scratch_address(dev, &scratch) != cudaSuccess) return SPV_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Start every call from a clear header: the error word, the self-test
    // flag and the streaming pass's work-item counter (bytes 0..15).  A caller
    // owning a workspace zero-fills it after a failed call; nobody can do that
    // for this array, so a counter left behind by a call whose finalize never
    // ran would otherwise make every later call skip work items.
    if (cudaMemsetAsync(scratch, 0, kHeaderClearBytes, st) != cudaSuccess) return SPV_ERR_CUDA;
    return spv::launch_chain_or_greedy(spv::chain_launch(a, scratch), st) == cudaSuccess ? SPV_OK : SPV_ERR_CUDA;
}

// Test hook, not part of the ABI (spv.h does not declare it): writes `value`
// into the scratch array's work-item counter on `stream`, the state a call
// that failed between its two launches would leave behind, so a test can
// check that the next call still starts from a clear header.
extern "C" spv_status spv_internal_noalloc_set_item_counter(unsigned long long value, void *stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPV_ERR_CUDA;
    void *scratch = nullptr;
    if (scratch_address(dev, &scratch) != cudaSuccess) return SPV_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // `value` lives on this stack frame: wait for the copy before returning.
    if (cudaMemcpyAsync(static_cast<unsigned char *>(scratch) + 8, &value, sizeof(value), cudaMemcpyHostToDevice,
                        st) != cudaSuccess)
        return SPV_ERR_CUDA;
    return cudaStreamSynchronize(st) == cudaSuccess ? SPV_OK : SPV_ERR_CUDA;
}

// nvfp4_quantize_experts_static_scratch: the routed activation quantiser for
// callers that cannot allocate device memory.
//
// Who needs it: code that runs where a cudaMalloc is not an option -- an
// inference server whose memory pool has already reserved the whole device
// for weights and KV cache (a further cudaMalloc fails or fragments it), and
// code on a latency-critical path that must not call cudaMalloc / cudaFree,
// which can synchronise the whole device.  Such callers still own their
// inputs and outputs; only the call's internal scratch moves here, into one
// fixed array per device that the library carries from load to exit.
#include <cstdio>
#include <mutex>

#include "../../include/nvfp4_moe.h"
#include "internal.h"

namespace {

// 4 MiB per device: the quantiser's scratch (status block, global scales,
// routing histograms and the routed-row map) for up to ~500,000 routed rows
// (tokens x k) with 128 experts.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;
static __device__ __align__(256) unsigned char g_quant_scratch[kStaticScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[256] = {nullptr};  // per device: the array's device address

// Device address of this device's copy of g_quant_scratch.  In host code the
// symbol itself is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, taken with the device current.
int scratch_address(void **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 256) {
        nvfp4::set_error("static scratch: no current CUDA device (%s)", cudaGetErrorString(e));
        return NVFP4_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_quant_scratch);
        if (e != cudaSuccess || !p) {
            nvfp4::set_error("static scratch: cudaGetSymbolAddress failed on device %d (%s)", dev,
                             cudaGetErrorString(e));
            return NVFP4_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return NVFP4_OK;
}

}  // namespace

extern "C" int nvfp4_quantize_experts_static_scratch(const uint16_t *x, int T, int H, const int32_t *topk_ids,
                                                     int k, int E, const float *input_scale, uint8_t *q_out,
                                                     uint8_t *sf_out, int sf_layout, int32_t *expert_offsets,
                                                     int32_t *perm, nvfp4_stream_t stream)
{
    // the workspace entry point's shape checks first, with its status codes,
    // so that a shape it refuses is refused here the same way
    const int shape_rc = nvfp4::quantize_shape_status(T, H, k, E);
    if (shape_rc != NVFP4_OK) return shape_rc;
    const size_t need = nvfp4_quantize_workspace_size(T, k, E);  // T * k fits an int after those checks
    if (need > kStaticScratchBytes) {
        nvfp4::set_error("static scratch: T=%d, k=%d, E=%d needs %zu bytes of scratch; the static array holds %zu "
                         "(use nvfp4_quantize_experts with a caller workspace)",
                         T, k, E, need, kStaticScratchBytes);
        return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    }
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != NVFP4_OK) return rc;
    // The call's first kernel resets the status block and counters that the
    // later kernels rely on; everything else in the scratch is written before
    // it is read, so stale contents from an earlier call do no harm.
    return nvfp4_quantize_experts(x, T, H, topk_ids, k, E, input_scale, q_out, sf_out, sf_layout, expert_offsets,
                                  perm, scratch, kStaticScratchBytes, stream);
}

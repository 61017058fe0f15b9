// MoE router on the device: softmax over the experts, top-k, renormalised.
//
// [page "Gemma 4 NVFP4 MoE 空输出", §矩阵融合 "MoE FFN": the routing result picks
// each token's experts and the expert outputs are summed with the routing
// weights; page "genesis-vllm-patches" (mlqm.cn), §3.3 patch P31: the softmax
// and top-k run on logits upcast to FP32.]
//
// One warp per token.  Lane l holds the logits of experts l, l+32, l+64, ...
// in registers (VPL = values per lane, a power of two with 32*VPL >= E), as
// order-preserving unsigned keys.  Selection takes k rounds of a warp arg-max
// over the experts not yet taken, ordered by (logit descending, expert index
// ascending), each round two warp reductions (redux.sync max of the key, then
// min of the index among the lanes that hold it): softmax is strictly
// increasing in the logit, so this is the probability order with ties to the
// lower index, and no exponential is needed to select.
//
// Weights: the full softmax renormalised over the k selected experts equals
// the softmax of the selected logits alone (the full normaliser cancels), so
// w_j = exp(l_j - l_top) / sum_i exp(l_i - l_top) over the k, in FP32 with
// the library's expf and an IEEE division.  The sum is a butterfly over the
// warp: every lane holds the same rounded total.

#include "internal.h"

namespace nvfp4 {

namespace {

template <typename In>
__device__ __forceinline__ float logit_f32(const In *p);
template <>
__device__ __forceinline__ float logit_f32<float>(const float *p)
{
    return __ldg(p);
}
template <>
__device__ __forceinline__ float logit_f32<uint16_t>(const uint16_t *p)
{
    return __uint_as_float((uint32_t)__ldg(p) << 16);  // BF16 -> FP32 is exact
}

// Order-preserving map of a finite FP32 value (or +-inf) to an unsigned key:
// larger value, larger key.  -0 is folded into +0 first (they compare equal
// as logits), and every key is at least 0x007FFFFF (-inf), so 0 can mark an
// expert that is taken or does not exist.
__device__ __forceinline__ uint32_t order_key(float v)
{
    const uint32_t b = __float_as_uint(v + 0.0f);  // -0 + +0 = +0 under round to nearest
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

template <int VPL, typename In>
__global__ void __launch_bounds__(256) router_topk_kernel(const In *__restrict__ logits, int T, int E, int k,
                                                          int32_t *__restrict__ topk_ids,
                                                          float *__restrict__ topk_w)
{
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    for (long long t = (long long)blockIdx.x * warps + (threadIdx.x >> 5); t < T; t += (long long)gridDim.x * warps) {
        const In *row = logits + t * E;
        uint32_t key[VPL];  // expert lane + 32 j; 0 once taken or beyond E
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int e = lane + 32 * j;
            key[j] = e < E ? order_key(logit_f32(row + e)) : 0u;
        }
        uint32_t mine_key = 0;  // lane r keeps the r-th selected (key, expert)
        int mine_e = 0;
        for (int r = 0; r < k; ++r) {
            uint32_t bk = 0;
            int bj = 0;
#pragma unroll
            for (int j = 0; j < VPL; ++j)  // ascending index: strict > keeps the lowest on ties
                if (key[j] > bk) {
                    bk = key[j];
                    bj = j;
                }
            // the largest key, then the lowest expert index holding it (e = 32 j + lane);
            // k <= E leaves an untaken expert in every round, so kmax > 0
            const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
            const uint32_t e = __reduce_min_sync(0xffffffffu, bk == kmax ? (uint32_t)(bj * 32 + lane) : 0xffffffffu);
            if ((uint32_t)lane == (e & 31u)) {
#pragma unroll
                for (int j = 0; j < VPL; ++j)
                    if (j == bj) key[j] = 0u;
            }
            if (lane == r) {
                mine_key = kmax;
                mine_e = (int)e;
            }
        }
        const float mine_v = key_value(mine_key);
        const float top = __shfl_sync(0xffffffffu, mine_v, 0);
        const float ex = lane < k ? expf(mine_v - top) : 0.0f;
        float s = ex;
#pragma unroll
        for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane < k) {
            topk_ids[t * k + lane] = mine_e;
            topk_w[t * k + lane] = ex / s;
        }
    }
}

template <typename In>
cudaError_t launch_router_typed(const In *logits, int T, int E, int k, int32_t *ids, float *w, cudaStream_t st)
{
    constexpr int kThreads = 256, kWarps = kThreads / 32;
    int sms = 0, dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    const long long want = ((long long)T + kWarps - 1) / kWarps;
    const int grid = (int)(want < (long long)sms * 8 ? want : (long long)sms * 8);
    const int vpl = E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : E <= 256 ? 8 : E <= 512 ? 16 : 32;
    switch (vpl) {
    case 1: router_topk_kernel<1, In><<<grid, kThreads, 0, st>>>(logits, T, E, k, ids, w); break;
    case 2: router_topk_kernel<2, In><<<grid, kThreads, 0, st>>>(logits, T, E, k, ids, w); break;
    case 4: router_topk_kernel<4, In><<<grid, kThreads, 0, st>>>(logits, T, E, k, ids, w); break;
    case 8: router_topk_kernel<8, In><<<grid, kThreads, 0, st>>>(logits, T, E, k, ids, w); break;
    case 16: router_topk_kernel<16, In><<<grid, kThreads, 0, st>>>(logits, T, E, k, ids, w); break;
    default: router_topk_kernel<32, In><<<grid, kThreads, 0, st>>>(logits, T, E, k, ids, w); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_topk(const void *logits, int bf16, int T, int E, int k, int32_t *ids, float *w,
                               cudaStream_t st)
{
    if (bf16) return launch_router_typed(static_cast<const uint16_t *>(logits), T, E, k, ids, w, st);
    return launch_router_typed(static_cast<const float *>(logits), T, E, k, ids, w, st);
}

}  // namespace nvfp4

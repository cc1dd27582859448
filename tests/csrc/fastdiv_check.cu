// Test-only: exhaustive check of the quantiser's division by the per-tile
// scale.  For every positive finite bf16 absmax A (hence every scale
// s = RN(A / 448) the quantising gather can produce on its fast path) and
// every finite bf16 x with |x| <= A, the e4m3 code that the kernel's 8-wide
// quantiser produces with the reciprocal + correction division must equal
// the code it produces with IEEE division.
#include "lmkv_fp8.cuh"

__global__ void fastdiv_exhaustive(unsigned long long* out) {
    const uint32_t a_bits = blockIdx.y + 1;                        // 0x0001 .. 0x7F7F
    const float amax = __uint_as_float(a_bits << 16);
    const float s = __fdiv_rn(amax, 448.0f);
    if (!(s >= lmkv::kFastDivMinScale)) return;                    // uniform per block
    const uint32_t base = (blockIdx.x * blockDim.x + threadIdx.x) * 8u;   // 8 inputs per thread
    uint32_t h[8];
    uint32_t in_mask = 0;
    for (int i = 0; i < 8; ++i) {
        const uint32_t xb = base + i;
        const float x = __uint_as_float(xb << 16);
        const bool in = isfinite(x) && fabsf(x) <= amax;
        h[i] = in ? xb : 0u;
        in_mask |= (in ? 1u : 0u) << i;
    }
    const uint4 v = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                               h[6] | (h[7] << 16));
    const uint2 cf = lmkv::quant_bf16x8<true>(v, lmkv::make_quant(s, true));
    const uint2 ci = lmkv::quant_bf16x8<false>(v, lmkv::make_quant(s, false));
    uint32_t diff = 0;
    for (int i = 0; i < 8; ++i) {
        const uint32_t bf = ((i < 4 ? cf.x : cf.y) >> (8 * (i & 3))) & 0xFFu;
        const uint32_t bi = ((i < 4 ? ci.x : ci.y) >> (8 * (i & 3))) & 0xFFu;
        if (((in_mask >> i) & 1u) && bf != bi) {
            ++diff;
            atomicCAS(&out[3], 0ull, ((unsigned long long)a_bits << 16) | (base + i));
        }
    }
    unsigned n_in = __popc(in_mask);
    for (int o = 16; o > 0; o >>= 1) {
        n_in += __shfl_xor_sync(0xFFFFFFFFu, n_in, o);
        diff += __shfl_xor_sync(0xFFFFFFFFu, diff, o);
    }
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&out[0], (unsigned long long)n_in);
        if (diff) atomicAdd(&out[1], (unsigned long long)diff);
    }
}

extern "C" int lmkv_test_fastdiv_exhaustive(unsigned long long* host_out) {
    unsigned long long* d = nullptr;
    if (cudaMalloc(&d, 4 * sizeof(unsigned long long)) != cudaSuccess) return 1;
    cudaMemset(d, 0, 4 * sizeof(unsigned long long));
    fastdiv_exhaustive<<<dim3(32, 0x7F7F), 256>>>(d);
    cudaError_t e = cudaDeviceSynchronize();
    cudaMemcpy(host_out, d, 4 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaFree(d);
    return e == cudaSuccess ? 0 : 2;
}

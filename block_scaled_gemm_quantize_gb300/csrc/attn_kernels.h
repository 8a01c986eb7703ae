// attn_kernels.h -- launch interface of the FP8 attention kernel (attn.cu),
// called by the C ABI layer after argument validation.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fp8bs {

struct AttnParams {
    int64_t seq_q, seq_k;     // query rows, keys (one sequence)
    int32_t hq, hkv;          // query heads, key/value heads (hq % hkv == 0)
    int32_t causal;
    float scale_log2;         // softmax scale * log2(e)
    const float* sq;          // [hq][seq_q]          Q scales (1x128 per token and head)
    const float* sk;          // [ceil(seq_k/128)][hkv] K scales (128 tokens x 128 per head)
    const float* sv;          // [ceil(seq_k/128)][hkv] V scales
    void* o;                  // bf16 [seq_q][ldo], head h at columns 128 h ..
    int64_t ldo;
    uint32_t idesc_s, idesc_o;
};

cudaError_t launch_fp8_attn_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const AttnParams& p, cudaStream_t st);
cudaError_t read_and_clear_attn_status(int* status);

}  // namespace fp8bs

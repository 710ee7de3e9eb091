// fg_mqa.cuh - host-visible parameters and launcher of the FP8 MQA-logits kernel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fg {

// Query tokens per kernel tile: the MMA's N is kMqaTokens x 64 heads.
constexpr int kMqaTokens = 4;

struct MqaParams {
    int S, T;                 // query tokens, kv tokens
    const float* kv_sf;       // [T]
    const float* weights;     // [S][64]
    const int32_t* ks;        // [S]
    const int32_t* ke;        // [S]
    float* out;               // [S][T]
    int clean;                // write -inf outside [ks, ke)
    int* status;
    unsigned long long timeout_ns;
    int pdl;
};

struct MqaMaps {
    CUtensorMap q;            // [S * 64][128] E4M3, boxes of kMqaTokens * 64 rows
    CUtensorMap kv;           // [T][128] E4M3, boxes of 128 rows
};

// grid CTAs, each walking groups of kMqaTokens query tokens blockIdx.x, blockIdx.x + grid, ...
cudaError_t launch_mqa(const MqaParams& p, const MqaMaps& maps, int grid, cudaStream_t stream);

}  // namespace fg

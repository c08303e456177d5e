// launch.h -- host-side launchers of the kernels (internal to libcpa).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/cpa.h"
#include "cpa_internal.h"

namespace cpa {

// Tensor maps for the tensor-core kernel (see attn_tc.cu).
struct TcMaps {
    CUtensorMap q;       // q      [T, H_q, d]   box (64, G, floor(128/G))
    CUtensorMap k_new;   // k_new  [T, H_kv, d]  box (64, 1, 128)
    CUtensorMap v_new;
    CUtensorMap k_pool;  // pool   [blocks, bs, H_kv, d]  box (64, 1, bs, 1)
    CUtensorMap v_pool;
};

cudaError_t launch_kv_write(const KvWriteArgs &a, int num_sms, cudaStream_t stream);
cudaError_t launch_rope(const RopeArgs &a, int num_sms, cudaStream_t stream);
cudaError_t launch_attn_simt(const AttnArgs &a, int dtype, cudaStream_t stream);
cudaError_t launch_attn_merge(const AttnArgs &a, int dtype, int num_split_reqs, cudaStream_t stream);
cudaError_t launch_attn_tc(const AttnArgs &a, const TcMaps &maps, cudaStream_t stream);
// two query tiles per unit (a.tiles_per_unit == 2), BF16 pools (attn_tc2.cu)
cudaError_t launch_attn_tc2(const AttnArgs &a, const TcMaps &maps, cudaStream_t stream);

}  // namespace cpa

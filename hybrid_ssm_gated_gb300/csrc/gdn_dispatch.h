// gdn_dispatch.h -- runtime dtype/shape -> kernel instantiation dispatch.
// Each dispatcher lives in its own translation unit so the instantiations
// compile in parallel.
#pragma once

#include <cuda_runtime.h>

#include "gdn_decode.cuh"
#include "gdn_prefill.cuh"
#include "gdn_replay_common.cuh"
#include "gdn_spec.cuh"

namespace gdn {

// Returns cudaErrorNotSupported when (state dtype, dk) has no instantiation.
cudaError_t dispatch_decode(int state_dtype, int dk, const DecodeArgs& a, cudaStream_t stream);

// tmax in {1, 4, 8}. too_big is set when the layout does not fit in shared memory.
cudaError_t dispatch_replay_f32(int dk, int tmax, ReplayArgs& a, cudaStream_t stream, bool& too_big);
cudaError_t dispatch_replay_bf16(int dk, int tmax, ReplayArgs& a, cudaStream_t stream, bool& too_big);
cudaError_t dispatch_replay_f16(int dk, int tmax, ReplayArgs& a, cudaStream_t stream, bool& too_big);
// An fp32 master checkpoint with a bf16 / fp16 read copy.
cudaError_t dispatch_replay_f32_bf16(int dk, int tmax, ReplayArgs& a, cudaStream_t stream, bool& too_big);
cudaError_t dispatch_replay_f32_f16(int dk, int tmax, ReplayArgs& a, cudaStream_t stream, bool& too_big);

// Mamba2 (RULE_MAMBA2): decode, and replay with one checkpoint (tmax in {1, 4, 8}).
cudaError_t dispatch_mamba2_decode(int state_dtype, int dk, const DecodeArgs& a, cudaStream_t stream);
cudaError_t dispatch_mamba2_replay_f32(int dk, int tmax, ReplayArgs& a, cudaStream_t stream, bool& too_big);
cudaError_t dispatch_mamba2_replay_bf16(int dk, int tmax, ReplayArgs& a, cudaStream_t stream, bool& too_big);
cudaError_t dispatch_mamba2_replay_f16(int dk, int tmax, ReplayArgs& a, cudaStream_t stream, bool& too_big);

// tmax in {4, 8}. too_big is set when the layout does not fit in shared memory.
cudaError_t dispatch_spec_f32(int dk, int tmax, SpecArgs& a, cudaStream_t stream, bool& too_big);
cudaError_t dispatch_spec_bf16(int dk, int tmax, SpecArgs& a, cudaStream_t stream, bool& too_big);
cudaError_t dispatch_spec_f16(int dk, int tmax, SpecArgs& a, cudaStream_t stream, bool& too_big);

// Prefill with a rounded write-back per chunk.
cudaError_t dispatch_prefill(int state_dtype, int dk, PrefillArgs& a, cudaStream_t stream);

// Rollback: pointer moves, checked against the window-length marker in each window's first record.
cudaError_t launch_rollback(int32_t* pos, const int32_t* ckpt_pos, float* ring_rec, const int32_t* slots,
                            const int32_t* accepted, int B, int Hv, int T, int L, int dv, int64_t num_slots,
                            int32_t* dev_err, cudaStream_t stream);

}  // namespace gdn

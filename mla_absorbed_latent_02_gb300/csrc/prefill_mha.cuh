// The prefill of long prompt chunks in the expanded (MHA) form: parameters
// and launchers of prefill_mha.cu (kept apart from the decode kernels' header).
#pragma once
#include "mla_kernels.cuh"

namespace mla {

// Long prompt chunks in the expanded (MHA) form: keys and values expanded from
// the latent once per sequence, then causal attention with 192-dim keys.
struct PrefillMhaParams {
  int B, H, T;             // sequences, heads, query tokens per sequence (the chunk)
  int max_len, ML;         // longest sequence allowed; rows per sequence in kv (max_len rounded up to 128)
  int paged, capacity, num_seqs, num_blocks, max_blocks;
  const int32_t* block_table;
  const int32_t* seq_lens;   // [B] tokens in the cache, the chunk's included
  const int32_t* q_pos;      // [B*T] RoPE positions of the queries
  const uint16_t* q_rope;    // [B*T, H, 64] bf16, before RoPE
  uint16_t* q_rot;           // [B*T, H, 64] bf16 after RoPE (workspace)
  uint16_t* kv;              // [B*ML, 2*H*128] bf16: K_nope of the H heads, then V (workspace)
  uint16_t* out;             // [B*T, H, 128] bf16
  const float2* rope;        // [max_pos, 32] cos/sin table
  int max_pos;
  float scale_log2;          // softmax scale * log2(e)
  int num_ctas;              // attention CTAs (one per SM, persistent)
  int* status;
};
cudaError_t launch_expand_kv(const CUtensorMap& tm_cache, const CUtensorMap& tm_wuk, const CUtensorMap& tm_wuv,
                             const CUtensorMap& tm_kvst, const PrefillMhaParams& p, cudaStream_t s);
cudaError_t launch_prefill_mha(const CUtensorMap& tm_qn, const CUtensorMap& tm_qr, const CUtensorMap& tm_kv,
                               const CUtensorMap& tm_cache, const PrefillMhaParams& p, cudaStream_t s);

}  // namespace mla

// Host-side launch interface between the C ABI (abi.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace skv {

constexpr int kMlaHeads = 64;
constexpr int kMlaDqk = 576;
constexpr int kMlaDv = 512;
constexpr int kMlaBlockRows = 64;   // top-k entries per block (split unit and pipeline step)

// Per-launch arguments of the sparse-MLA decode kernel (split or direct epilogue).
struct MlaArgs {
  const uint8_t* kv;    // [n_kv][576] bf16 rows of 1152 B
  const int32_t* idx;   // [s_q][topk]
  int s_q;
  int topk;
  int n_kv;
  int num_splits;       // uniform schedule: splits per token (1 for the direct path)
  int num_blocks;       // ceil(topk / 64): 64-row blocks per token
  int dim_groups;       // uniform schedule: CTAs per (token, split) job (1, 2 or 4); CTA
                        // g of a job computes the same scores and softmax and the
                        // output dims [512 g / dim_groups, 512 (g + 1) / dim_groups)
  int sched;            // 0: (token, split) jobs, grid s_q * num_splits * dim_groups;
                        // 1: balanced, the s_q * num_blocks blocks cut into num_ctas
                        //    near-equal contiguous ranges, one per CTA (grid num_ctas)
  int num_ctas;         // balanced schedule: CTAs (<= s_q * num_blocks)
  int direct_whole;     // a job that covers a whole token writes the final output
                        // (sink, cast, LSE, amax) instead of a partial
  int tail_first;       // uniform schedule with tail_splits > 0: tokens 0 .. tail_first - 1
  int tail_splits;      // run whole on CTAs 0 .. tail_first - 1; tokens tail_first .. s_q - 1
                        // are cut into tail_splits splits, CTA tail_first + k running split
                        // k % tail_splits of tail token k / tail_splits, whose partial goes to
                        // slot (split, tail token) of the workspace (needs num_splits ==
                        // dim_groups == 1); 0: no tail
  int check_idx;        // 1: a loader that meets an index outside {-1} and [0, n_kv) sets
                        // status bit 0x10 (the row stays masked either way)
  int tail_dgroups;     // uniform schedule, tail_splits == 0: tokens tail_first .. s_q - 1 run
                        // whole on tail_dgroups (2 or 4) CTAs each, CTA tail_first + k taking
                        // dim group k % tail_dgroups of tail token k / tail_dgroups and
                        // writing its final rows (needs num_splits == dim_groups == 1); 0: no
  float scale_log2;     // sm_scale * log2(e)
  // Partial workspace: [slot][s_q][64][512] and [slot][s_q][64]. Uniform: slot =
  // the split. Balanced: slot = a piece's place among the pieces of its token
  // (a token cut by range boundaries); whole tokens write their final rows.
  float* o_acc;         // fp32, or bf16 values when partial_bf16
  float* lse_acc;
  int partial_bf16;     // O partials stored as bf16 (LSE partials stay fp32)
  // direct path: final output
  void* out;            // [s_q][64][512] of out_dtype
  int out_dtype;
  float inv_scale;
  float* lse_out;       // [s_q][64] or null
  const float* sink;    // [64] or null
  float* amax;          // scalar or null (zeroed by the launcher)
  uint32_t* status;     // device status words [2]
  uint64_t wait_limit_ns;   // a pipeline wait that runs longer records a timeout and aborts the CTA
  uint64_t drain_limit_ns;  // how long an aborting CTA waits for its own copies and MMAs in flight
};

// Balanced schedule arithmetic, shared by the host and the decode kernel: U
// units (64-row blocks, token-major) cut into P contiguous ranges, the first
// U % P of them one unit longer. Requires 1 <= P <= U.
__host__ __device__ inline int bal_begin(int p, int U, int P) {
  const int base = U / P, rem = U % P;
  return p * base + (p < rem ? p : rem);
}
// The range (CTA) that holds unit u.
__host__ __device__ inline int bal_cta_of(int u, int U, int P) {
  const int base = U / P, rem = U % P;
  const int big = rem * (base + 1);
  return u < big ? u / (base + 1) : rem + (u - big) / base;
}

// Dynamic shared memory the MLA decode kernel needs.
int mla_decode_smem_bytes();
// One-time per-device set-up (shared-memory opt-in of the kernels); called by the
// ABI the first time it sees a device, outside any stream capture.
cudaError_t prepare_mla_kernels();
cudaError_t prepare_sdpa_kernels();

// tm_q: Q viewed as 2-D [s_q*64 rows][576] bf16, box 64x64, 128B swizzle.
cudaError_t launch_mla_decode(const CUtensorMap& tm_q, const MlaArgs& a, cudaStream_t stream);

// Log-sum-exp combine over `rows` output rows of width d (512 or 128).
struct CombineArgs {
  const float* o_acc;   // [S][rows][d], fp32 or (partial_bf16) bf16 values
  const float* lse_acc; // [S][rows]
  int partial_bf16;
  int num_splits;
  int rows;             // tokens * heads
  int heads;            // head index = row % heads (for the sink)
  int d;
  const float* sink;    // [heads] or null
  void* out;
  int out_dtype;
  float inv_scale;
  float* lse_out;       // [rows] or null
  float* amax;          // scalar or null
  // Balanced sparse-MLA schedule (bal_ctas > 0): row r belongs to token r / heads,
  // whose split count is the number of CTA ranges its bal_nb blocks fall in (the
  // blocks of all tokens, bal_units of them, cut into bal_ctas ranges); a token in
  // one range was finished by the decode kernel and is left alone.
  int bal_nb, bal_units, bal_ctas;
  int num_sms;          // SMs of the device (caps the grid; 0: one CTA per 8 items)
  int sparse_splits;    // most split slots of most rows are empty (LSE -inf): load a
                        // slice only once its weight is known to be non-zero
};
// zero_amax: clear *amax first (a memset on the stream); pdl: launch as a
// programmatic dependent of the preceding kernel on the stream.
cudaError_t launch_combine(const CombineArgs& a, bool zero_amax, bool pdl, cudaStream_t stream);

// Bounded-wait self test: one CTA waits on a barrier nobody arrives on.
cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t stream);

// Dense FP8 split-KV SDPA decode.
struct SdpaArgs {
  const uint8_t* q;             // [total_q][h_q][128] e4m3
  const int32_t* cu_q;          // [batch+1]
  const int32_t* cu_kv;         // [batch+1]
  const float* descale_q;       // device scalars or null
  const float* descale_k;
  const float* descale_v;
  int batch, h_q, h_kv, total_q, num_splits;
  int adaptive;                 // per-sequence split counts (<= num_splits) from the KV lengths
  int num_sms;                  // SM count the adaptive rule spreads the work over
  float scale_log2;
  float* o_acc;                 // split path [S][total_q][h_q][128]
  float* lse_acc;               // [S][total_q][h_q]
  void* out;                    // direct path [total_q][h_q][128]
  int out_dtype;
  float inv_scale;
  float* lse_out;
  float* amax;
  uint32_t* status;
  uint64_t wait_limit_ns;   // as in MlaArgs
  uint64_t drain_limit_ns;
};
int sdpa_decode_smem_bytes();
// tm_q: Q viewed as 3-D [total_q][h_q][128] e4m3, box {128 d, group heads, 64/group tokens}.
// tm_k / tm_v: K and V viewed as 3-D [total_kv][h_kv][128] e4m3, box {128 d, 1 head, 128 keys}.
cudaError_t launch_sdpa_decode(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                               const SdpaArgs& a, bool direct, cudaStream_t stream);

}  // namespace skv

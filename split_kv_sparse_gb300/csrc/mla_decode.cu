// Split-KV sparse-MLA decode kernel for sm_103a (tcgen05 MMAs, TMEM accumulators,
// cp.async row gathers).
//
// What one job computes (FlashMLA PR #25, "What changes"): the job (query token
// t, a range [row0, row1) of its top-k entries) gathers those rows of the shared
// latent KV cache and produces, for each of the 64 heads,
//   a partial:   O = sum_r e^{s_r} V_r / sum_r e^{s_r} (fp32) and the log2 LSE, or
//   final rows:  the same O with the attention sink folded into the denominator,
//                cast to fp32 / bf16 / e4m3, plus LSE and amax (a job that
//                covers all of its token's entries).
//
// Which jobs a CTA runs (the schedule):
//   uniform   one (token, split) job per CTA: split s of S takes a near-equal run
//             of 64-row blocks, remainder to the leading splits (cuDNN-frontend
//             PR #768, SM120 FP8 commit). With dim_groups D > 1 a job runs on D
//             CTAs that compute the same scores and softmax and each write
//             512/D of the output dims; grid s_q * S * D.
//   balanced  the s_q * nb blocks of all tokens, token-major, are cut into
//             num_ctas near-equal contiguous ranges, one per CTA, so every SM
//             walks the same number of rows whatever s_q is. A CTA runs one job
//             per token its range touches. A whole token gets its final rows; each
//             piece of a token cut by range boundaries is a partial in the split
//             layout, slot = the piece's place among its token's pieces, and the
//             combine folds them by the log-sum-exp rule ("The Split-K Dispatch",
//             "The LSE Combine Strategy"). Only on request: measured slower
//             than the uniform grid at every s_q tried (the planner's notes).
// The kernel is compiled once per schedule, so the uniform one carries none of
// the job switching.
//
// Layout of the work (256 threads, 64 gathered rows per step; the steps of all
// of a CTA's jobs form one sequence, one pipeline over a ring of two 64-row
// halves; the row gathers and the MMA issue run on across job boundaries):
//   warps 0-1  row gathers: warp w copies rows 32w..32w+31 of the step; lane i
//              takes 16-byte piece i mod 8 of every 64-dim chunk of rows
//              32w + 4m + i/8 (m = 0..7), so one warp instruction copies four
//              whole 128-byte lines; each copy is one instruction with constant
//              offsets on both addresses, into the 128-byte-swizzled layout. An
//              invalid index copies zeros and reads nothing. Completion:
//              cp.async.mbarrier.arrive.
//   warp 2     Q of each job by TMA (9 tiles of 64 heads x 64 dims), once the
//              previous job's last QK has finished with the buffer (a barrier
//              with one phase per job: a waiter on an mbarrier parity must never
//              fall two phases behind, which a per-step barrier would allow here).
//   warp 3     tcgen05 issue (one thread), all descriptors precomputed:
//                S[64 heads x 64 rows]  = Q . K_half^T                (M=64, N=64, K=576)
//                O^T[512 x 64 heads]   += V_half^T . P_hi^T, then . P_lo^T (4 x (M=128, N=64, K=64) each)
//              V is read straight out of the gathered rows as an MN-major
//              operand; Q, K and P^T are K-major; all tiles use the 128-byte
//              swizzle. Each QK is one unbroken run of its 36 MMAs.
//   warps 4-7  softmax: an M=64 accumulator keeps head 16w+i in lane i of TMEM
//              sub-partition w, so warp 4+w owns heads 16w..16w+15; its lanes
//              0-15 take rows 0-31 and lanes 16-31 rows 32-63 of the step (one
//              16x32bx2 TMEM load). A head's running max and row sum live in two
//              lanes of one warp; only a rescale of O^T (rare, lazy) is shared
//              with the other warps, through a per-step barrier that is arrived
//              on early and waited on late. P_hi is published before P_lo, whose
//              one buffer must first be released by the previous PV. At the end
//              of each job: the epilogue, straight from TMEM to global memory;
//              for a job followed by another (balanced schedule) it runs after
//              the next job's first softmax step, while that step's PV writes
//              its O^T tiles 0 and 1 to a second place (tile_col) and waits for
//              the epilogue to have read tiles 2 and 3.
//
// Precision: p = 2^(x - m_ref) is stored as P_hi = p truncated to bf16 and
// P_lo = bf16(p - P_hi); the PV product uses both, so P enters O with ~2^-15
// relative error instead of the 2^-8 of a single bf16. The fp32 sum of p (the
// softmax denominator, and the LSE) is kept per thread and reduced at the end of
// the job; it matches the P the product used to the same ~2^-15.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"
#include "softmax_util.cuh"

namespace skv {
namespace {

constexpr int kThreads = 256;
constexpr int kLoaders = 64;                        // warps 0-1
constexpr int kChunks = 9;                          // 576 dims = 9 column chunks of 64 (128 B)
constexpr int kSlotBytes = 16384;                   // one column chunk of both halves
constexpr int kHalfBytes = 8192;                    // one column chunk of one 64-row half
constexpr int kQChunkBytes = 8192;                  // 64 heads x 128 B
constexpr int kRingBytes = kChunks * kSlotBytes;    // 147456
constexpr int kQBytes = kChunks * kQChunkBytes;     // 73728
constexpr int kRowBytes = kMlaDqk * 2;              // 1152

// Shared memory map. The dynamic shared memory base is 1024-byte aligned (the
// kernel checks it and refuses to run otherwise), so no slack is reserved.
constexpr int kOffRing = 0;
constexpr int kOffQ = kOffRing + kRingBytes;        // 147456
constexpr int kOffPlo = kOffQ + kQBytes;            // 221184: P_lo^T, 64 heads x 64 rows bf16
constexpr int kOffBars = kOffPlo + kHalfBytes;      // 229376
constexpr int kOffMisc = kOffBars + 256;            // [0] tmem base, [1] abort flag,
                                                    // [4..11] rescale masks [2][4], [12..15] failure flags
constexpr int kOffAlpha = kOffMisc + 128;           // float[2][64] rescale factors by step parity
constexpr int kOffHead = kOffAlpha + 512;           // float[2][2][64] per-head epilogue scalars by job parity
constexpr int kSmemBytes = kOffHead + 1024;         // 231296

// The ring half of each step is filled and released in two chunk groups: A =
// column chunks 0-3 (the V dims of O^T tiles 0 and 1) and B = chunks 4-8 (tiles
// 2 and 3 and the RoPE chunk, which holds P_hi once the scores are computed). A
// group is refilled as soon as the PV MMAs that read it are done, so the rows of
// step g + 2 start landing while PV(g) still runs.
enum {
  B_QFULL = 0, B_FULLA0, B_FULLA1, B_FULLB0, B_FULLB1, B_EMPTYA0, B_EMPTYA1, B_EMPTYB0, B_EMPTYB1,
  B_SFULL0, B_SFULL1, B_PHI0, B_PHI1, B_PLO0, B_PLO1, B_PVDONE, B_DRAIN, B_XCH0, B_XCH1, B_OFREE2,
  B_OFREE3, B_QFREE, B_OT0, B_OT1, B_OT2, B_OT3, kNumBars
};
constexpr int kGroupSplit = 4;                      // chunks [0, 4) form group A, [4, 9) group B
static_assert(kNumBars * 8 <= 256, "barrier area");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 256;                    // S buffers at columns 256 and 320
constexpr uint32_t kTmemAlt = 384;                  // tiles 0 and 1 of O^T for odd jobs: columns 384..511
constexpr float kRescaleThreshold = 8.0f;           // p = 2^(x - m_ref) <= 256 between rescales
constexpr float kLog2e = 1.4426950408889634f;

// Wait sites reported in the status word when a bounded wait runs out.
enum : uint32_t {
  W_PROD_EMPTY = 1, W_MMA_Q, W_MMA_STALL, W_SM_S, W_SM_PV, W_SM_PV_EPI, W_DRAIN_MMA, W_SM_X, W_PROD_Q,
  W_DRAIN_Q = 11
};

// 128-byte-swizzled byte offset of the 16-byte piece `piece` (0-7) of row `row`
// inside a tile of 128-byte rows grouped in 1024-byte, 8-row atoms.
__device__ __forceinline__ int sw128(int row, int piece) {
  return (row >> 3) * 1024 + (row & 7) * 128 + ((piece ^ (row & 7)) << 4);
}

// The copies of one lane for one row: its 16-byte piece of each 64-dim chunk
// C .. kEnd-1. `dst` is the piece's swizzled place in chunk 0, `src` its bytes
// in chunk 0; chunk c adds c * kSlotBytes to the one and c * 128 to the other.
template <int C, int kEnd>
__device__ __forceinline__ void copy_row_chunks(uint32_t dst, const uint8_t* src, uint32_t sz) {
  if constexpr (C < kEnd) {
    cp_async_16_off2<C * kSlotBytes, C * 128>(dst, src, sz);
    copy_row_chunks<C + 1, kEnd>(dst, src, sz);
  }
}

enum : int { J_FINAL = 0, J_PARTIAL = 1 };

// One job of a CTA: token t, top-k entries [row0, row1) in nsteps steps of 64.
//   J_FINAL    final rows of token t;
//   J_PARTIAL  a partial at workspace rows out_row .. + 63: a (token, split) job
//              of the uniform schedule, or a piece of a token cut by the balanced
//              schedule (slot = the piece's place among its token's pieces).
struct Job {
  int t, row0, row1, nsteps, kind, slot;
  int q0, nq;   // the 128-dim tiles of O^T this CTA computes: q0 .. q0+nq-1
  size_t out_row;
};

template <int kSched>
__device__ __forceinline__ int num_jobs(const MlaArgs& a) {
  if (kSched == 0) return 1;
  const int U = a.s_q * a.num_blocks, P = a.num_ctas, p = blockIdx.x;
  const int u0 = bal_begin(p, U, P), u1 = bal_begin(p + 1, U, P);
  return (u1 - 1) / a.num_blocks - u0 / a.num_blocks + 1;
}

template <int kSched>
__device__ __forceinline__ Job job_at(const MlaArgs& a, int j) {
  Job r;
  if (kSched == 0 && a.tail_dgroups > 0 && static_cast<int>(blockIdx.x) >= a.tail_first) {
    // a tail token run whole on tail_dgroups CTAs, each with its share of the dims
    const int D = a.tail_dgroups;
    const int k = static_cast<int>(blockIdx.x) - a.tail_first;
    const int tt = k / D, dg = k - tt * D;
    r.nq = 4 / D;
    r.q0 = dg * r.nq;
    r.t = a.tail_first + tt;
    r.row0 = 0;
    r.row1 = a.topk;
    r.nsteps = a.num_blocks;
    r.kind = J_FINAL;
    r.slot = 0;
    r.out_row = static_cast<size_t>(r.t) * kMlaHeads;
  } else if (kSched == 0 && a.tail_splits > 0 && static_cast<int>(blockIdx.x) >= a.tail_first) {
    // a piece of a token of the tail: near-equal block runs as for S splits
    const int S = a.tail_splits, nt = a.s_q - a.tail_first;
    const int k = static_cast<int>(blockIdx.x) - a.tail_first;
    const int tt = k / S, s = k - tt * S;
    r.nq = 4;
    r.q0 = 0;
    const int base = a.num_blocks / S, rem = a.num_blocks - base * S;
    const int blk0 = s * base + min(s, rem), nblk = base + (s < rem ? 1 : 0);
    r.t = a.tail_first + tt;
    r.row0 = min(blk0 * kMlaBlockRows, a.topk);
    r.row1 = min((blk0 + nblk) * kMlaBlockRows, a.topk);
    r.nsteps = (r.row1 - r.row0 + kMlaBlockRows - 1) / kMlaBlockRows;
    r.kind = J_PARTIAL;
    r.slot = s;
    r.out_row = (static_cast<size_t>(s) * nt + tt) * kMlaHeads;
  } else if (kSched == 0) {
    const int S = a.num_splits, D = a.dim_groups;
    const int job = static_cast<int>(blockIdx.x) / D, dg = static_cast<int>(blockIdx.x) - job * D;
    const int t = job / S, s = job - t * S;
    r.nq = 4 / D;
    r.q0 = dg * r.nq;
    const int base = a.num_blocks / S, rem = a.num_blocks - base * S;
    const int blk0 = s * base + min(s, rem), nblk = base + (s < rem ? 1 : 0);
    r.t = t;
    r.row0 = min(blk0 * kMlaBlockRows, a.topk);
    r.row1 = min((blk0 + nblk) * kMlaBlockRows, a.topk);
    r.nsteps = (r.row1 - r.row0 + kMlaBlockRows - 1) / kMlaBlockRows;
    r.kind = (a.direct_whole && S == 1) ? J_FINAL : J_PARTIAL;
    r.slot = s;
    r.out_row = r.kind == J_FINAL ? static_cast<size_t>(t) * kMlaHeads
                                  : (static_cast<size_t>(s) * a.s_q + t) * kMlaHeads;
  } else {
    const int nb = a.num_blocks, U = a.s_q * nb, P = a.num_ctas, p = blockIdx.x;
    const int u0 = bal_begin(p, U, P), u1 = bal_begin(p + 1, U, P);
    const int t = u0 / nb + j;
    const int b0 = max(u0, t * nb) - t * nb, b1 = min(u1, (t + 1) * nb) - t * nb;
    r.t = t;
    r.row0 = b0 * kMlaBlockRows;
    r.row1 = min(b1 * kMlaBlockRows, a.topk);
    r.nsteps = b1 - b0;
    r.kind = (b0 == 0 && b1 == nb) ? J_FINAL : J_PARTIAL;
    r.slot = p - bal_cta_of(t * nb, U, P);
    r.q0 = 0;
    r.nq = 4;
    r.out_row = r.kind == J_FINAL ? static_cast<size_t>(t) * kMlaHeads
                                  : (static_cast<size_t>(r.slot) * a.s_q + t) * kMlaHeads;
  }
  return r;
}

// The steps of a CTA, in order over all of its jobs: step g gathers top-k
// entries [r0, r1) of token t and belongs to job `job` (the CTA's job index),
// of which it may be the first and/or the last step.
struct Step {
  int t, r0, r1, job;
  bool first, last;
};

template <int kSched>
__device__ __forceinline__ Step step_at(const MlaArgs& a, const Job& j0, int u0, int total, int g) {
  Step s;
  if (kSched == 0) {
    s.t = j0.t;
    s.r0 = j0.row0 + kMlaBlockRows * g;
    s.r1 = min(s.r0 + kMlaBlockRows, j0.row1);
    s.job = 0;
    s.first = g == 0;
    s.last = g == total - 1;
  } else {
    const int nb = a.num_blocks, u = u0 + g;
    s.t = u / nb;
    const int b = u - s.t * nb;
    s.r0 = b * kMlaBlockRows;
    s.r1 = min(s.r0 + kMlaBlockRows, a.topk);
    s.job = s.t - u0 / nb;
    s.first = g == 0 || b == 0;
    s.last = g == total - 1 || b == nb - 1;
  }
  return s;
}

// TMEM column of O^T tile q for the CTA's job jj: tiles 0 and 1 alternate
// between columns 0..127 and 384..511 by job parity, so a job's first PV can
// write them while the epilogue of the job before still reads that job's
// tiles (which it takes in the order 2, 3, 0, 1).
__device__ __forceinline__ uint32_t tile_col(int q, int jj) {
  return 64u * static_cast<uint32_t>(q) + ((q < 2 && (jj & 1)) ? kTmemAlt : 0u);
}

// 4x4 transpose of 32-bit words across the four lanes whose lane bits `b` and
// `2b` differ (lane i holds m[0..3]; afterwards it holds word i of each of the
// four lanes, in lane order). Two butterfly stages of two exchanges each.
__device__ __forceinline__ void transpose4_words(uint32_t (&m)[4], int lane, int b) {
  const bool hi1 = (lane & (2 * b)) != 0, hi0 = (lane & b) != 0;
#pragma unroll
  for (int r = 0; r < 2; ++r) {   // distance 2 in the quad: swap the off-diagonal 2x2 blocks
    const uint32_t snd = hi1 ? m[r] : m[r + 2];
    const uint32_t rcv = __shfl_xor_sync(0xffffffffu, snd, 2 * b);
    if (hi1) m[r] = rcv; else m[r + 2] = rcv;
  }
#pragma unroll
  for (int r = 0; r < 4; r += 2) {   // distance 1: swap within each 2x2 block
    const uint32_t snd = hi0 ? m[r] : m[r + 1];
    const uint32_t rcv = __shfl_xor_sync(0xffffffffu, snd, b);
    if (hi0) m[r] = rcv; else m[r + 1] = rcv;
  }
}

// Final rows of one O^T tile column set, cast and stored; returns max |v| of
// this thread's values. Lane l of the warp holds v[c] = O[head c][d0 + l] for the
// 64 heads; d0 (a multiple of 32) is the same for the whole warp, and every lane
// of the warp calls this together. fp32 rows are stored as they are (each store
// instruction covers 128 contiguous bytes of one head). bf16 and e4m3 codes are
// first moved across lanes so that each lane holds 16 contiguous bytes of one
// head row, stored with one 16-byte store per head and half-row group.
// `rows`: the token's [64 heads][512] rows of element type `dtype` (0 fp32, 1
// bf16, 2 e4m3 scaled by inv_scale).
__device__ __forceinline__ float store_rows(void* rows, int dtype, float inv_scale, int d0, int lane,
                                            const float (&v)[64]) {
  float m = 0.f;
#pragma unroll
  for (int c = 0; c < 64; ++c) m = fmaxf(m, fabsf(v[c]));
  const size_t row0 = static_cast<size_t>(d0);   // head 0, dim d0
  if (dtype == 0) {
    float* st = static_cast<float*>(rows) + row0 + lane;
#pragma unroll
    for (int c = 0; c < 64; ++c) st[c * kMlaDv] = v[c];
  } else if (dtype == 1) {
    // w[k]: heads 2k, 2k+1 at dim d0 + lane. Lane pairs swap halves, so lane
    // 2i+j holds head 2k+j at dims 2i, 2i+1; then the four lanes 8h+2i'+j
    // (i' = 0..3) transpose groups of four words, so lane 8h+2i'+j holds, for k
    // = 4G+i', head 2k+j at dims 8h .. 8h+7.
    const bool odd = (lane & 1) != 0;
#pragma unroll
    for (int G = 0; G < 8; ++G) {
      uint32_t w[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int k = 4 * G + r;
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        const uint32_t x = *reinterpret_cast<const uint32_t*>(&h2);
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, 1);
        // even lane: (own head 2k, partner's head 2k); odd: (partner's 2k+1, own 2k+1)
        w[r] = odd ? __byte_perm(x, y, 0x3276) : __byte_perm(x, y, 0x5410);
      }
      transpose4_words(w, lane, 2);
      const int ip = (lane >> 1) & 3, j = lane & 1, hq = lane >> 3;
      const int head = 2 * (4 * G + ip) + j;
      __nv_bfloat16* st = static_cast<__nv_bfloat16*>(rows) + row0 + static_cast<size_t>(head) * kMlaDv + 8 * hq;
      *reinterpret_cast<uint4*>(st) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    // w[k]: heads 4k .. 4k+3 at dim d0 + lane, one byte each. A 4x4 byte
    // transpose in each lane quad gives lane 4i+j head 4k+j at dims 4i .. 4i+3;
    // then the four lanes 16h+4i'+j transpose groups of four words, so lane
    // 16h+4i'+j holds, for k = 4G+i', head 4k+j at dims 16h .. 16h+15.
    const int j = lane & 3;
    const uint32_t sel1 = (j & 2) ? 0x3276u : 0x5410u;
    const uint32_t sel2 = (j & 1) ? 0x3715u : 0x6240u;
#pragma unroll
    for (int G = 0; G < 4; ++G) {
      uint32_t w[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int k = 4 * G + r;
        const uint32_t c01 = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * k] * inv_scale, v[4 * k + 1] * inv_scale),
                                                      __NV_SATFINITE, __NV_E4M3);
        const uint32_t c23 = __nv_cvt_float2_to_fp8x2(
            make_float2(v[4 * k + 2] * inv_scale, v[4 * k + 3] * inv_scale), __NV_SATFINITE, __NV_E4M3);
        uint32_t x = (c01 & 0xFFFFu) | (c23 << 16);
        x = __byte_perm(x, __shfl_xor_sync(0xffffffffu, x, 2), sel1);
        w[r] = __byte_perm(x, __shfl_xor_sync(0xffffffffu, x, 1), sel2);
      }
      transpose4_words(w, lane, 4);
      const int ip = (lane >> 2) & 3, hq = lane >> 4;
      const int head = 4 * (4 * G + ip) + j;
      uint8_t* st = static_cast<uint8_t*>(rows) + row0 + static_cast<size_t>(head) * kMlaDv + 16 * hq;
      *reinterpret_cast<uint4*>(st) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  return m;
}

// Final rows of token t (the call's output, its dtype and scale).
__device__ __forceinline__ float store_final(const MlaArgs& a, int t, int d0, int lane, const float (&v)[64]) {
  const size_t esz = a.out_dtype == 0 ? 4 : (a.out_dtype == 1 ? 2 : 1);
  return store_rows(static_cast<uint8_t*>(a.out) + static_cast<size_t>(t) * kMlaHeads * kMlaDv * esz, a.out_dtype,
                    a.inv_scale, d0, lane, v);
}

// kSched: 0 = uniform (one job per CTA), 1 = balanced (a run of jobs per CTA);
// one instance per schedule keeps the uniform one free of the job switching.
template <int kSched>
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const MlaArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- jobs and steps: the same decode in every role -----------------------
  const int njobs = num_jobs<kSched>(a);
  const Job j0 = job_at<kSched>(a, 0);
  int u0 = 0, total = j0.nsteps;   // the CTA's first 64-row block (balanced) and its step count
  if (kSched != 0) {
    const int U = a.s_q * a.num_blocks;
    u0 = bal_begin(blockIdx.x, U, a.num_ctas);
    total = bal_begin(blockIdx.x + 1, U, a.num_ctas) - u0;
  }

  if (j0.nsteps == 0) {
    // A split with no block of its own (uniform schedule only): O = 0 over this
    // CTA's dims, LSE = -inf (written by the CTA of the first dims).
    grid_launch_dependents();
    grid_dependency_wait();   // the preceding kernel may still read this workspace
    const int per_head = 32 * j0.nq;   // groups of 4 values of one head row this CTA owns
    if (a.partial_bf16) {
      uint2* o = reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.o_acc) + j0.out_row * kMlaDv);
      for (int i = threadIdx.x; i < kMlaHeads * per_head; i += kThreads) {
        const int h = i / per_head;
        o[h * (kMlaDv / 4) + 32 * j0.q0 + (i - h * per_head)] = make_uint2(0u, 0u);
      }
    } else {
      float4* o = reinterpret_cast<float4*>(a.o_acc + j0.out_row * kMlaDv);
      for (int i = threadIdx.x; i < kMlaHeads * per_head; i += kThreads) {
        const int h = i / per_head;
        o[h * (kMlaDv / 4) + 32 * j0.q0 + (i - h * per_head)] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (j0.q0 == 0 && threadIdx.x < kMlaHeads) a.lse_acc[j0.out_row + threadIdx.x] = -INFINITY;
    return;
  }
  if ((sbase & 1023u) != 0) {
    // the swizzled tiles need a 1024-byte aligned base; report and do nothing
    grid_launch_dependents();
    if (threadIdx.x == 0) atomicOr(&a.status[0], 4u);
    return;
  }

  auto bar = [&](int i) -> uint32_t { return sbase + kOffBars + 8 * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile uint32_t* xch = reinterpret_cast<volatile uint32_t*>(misc + 4);   // [2][4] rescale masks
  volatile int* fin = reinterpret_cast<volatile int*>(misc + 12);             // [4] per-warp failure flags
  float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
  float* hs = reinterpret_cast<float*>(smem + kOffHead);   // [job parity][2][64] per-head scalars
  const WaitCtx wc{a.wait_limit_ns, a.status, abort_flag};

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(B_FULLA0 + i), kLoaders);   // one cp.async completion arrival per loader thread
      mbar_init(bar(B_EMPTYA0 + i), 1);         // one MMA commit
    }
    mbar_init(bar(B_SFULL0), 1);
    mbar_init(bar(B_SFULL1), 1);
    mbar_init(bar(B_PHI0), 4);             // one arrival per softmax warp
    mbar_init(bar(B_PHI1), 4);
    mbar_init(bar(B_PLO0), 4);
    mbar_init(bar(B_PLO1), 4);
    mbar_init(bar(B_PVDONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_XCH0), 4);
    mbar_init(bar(B_XCH1), 4);
    mbar_init(bar(B_OFREE2), 4);           // a job's O^T tile 2 read by the epilogue, per softmax warp
    mbar_init(bar(B_OFREE3), 4);           // and its tile 3
    mbar_init(bar(B_QFREE), 1);            // a job's last QK has completed: its Q buffer is free
    for (int i = 0; i < 4; ++i) mbar_init(bar(B_OT0 + i), 1);   // O^T tile i of a job is complete
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 3) {
    tmem_alloc(smem_u32(misc), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  // A programmatic dependent (the combine, or the next call) may begin
  // launching now; it waits for this whole grid before it touches memory.
  grid_launch_dependents();
  // This grid may itself have started early, behind the preceding kernel on the
  // stream: everything above touched only this CTA's own resources; from here
  // on it reads its inputs and writes its outputs, so that kernel must be done.
  grid_dependency_wait();

  // The first row indices: a loader lane takes row 32w + lane of step 0; a
  // softmax lane takes rows lane and lane + 32.
  int pre0 = -1, pre1 = -1;
  {
    const int32_t* idx0 = a.idx + static_cast<size_t>(j0.t) * a.topk;
    int r = -1, r2 = -1;
    if (warp < 2) {
      r = j0.row0 + 32 * warp + lane;
    } else if (warp >= 4) {
      r = j0.row0 + lane;
      r2 = r + 32;
    }
    if (r >= 0 && r < j0.row1) pre0 = __ldg(idx0 + r);
    if (r2 >= 0 && r2 < j0.row1) pre1 = __ldg(idx0 + r2);
  }

  if (warp < 2) {
    // ====================================================== row gathers ===
    const int pc = lane & 7;                       // this lane's 16-byte piece of a chunk
    const int ro = lane >> 3;                      // and its row within each group of 4
    // index of row 32w + lane of step g (any job of the CTA), -1 past the rows
    auto fetch = [&](int g) -> int {
      if (g >= total) return -1;
      const Step s = step_at<kSched>(a, j0, u0, total, g);
      const int r = s.r0 + 32 * warp + lane;
      return r < s.r1 ? __ldg(a.idx + static_cast<size_t>(s.t) * a.topk + r) : -1;
    };
    // Rows two steps ahead are requested into L2 as soon as their index is
    // known: with two ring halves a step's rows are copied only once the step
    // two before has finished with its half, so without this their DRAM
    // latency would sit on the loop's critical chain. One prefetch per
    // 128-byte line from the load/store path (a bulk prefetch per row goes
    // through the copy engine, which takes the requests one at a time). The
    // steps run on across the CTA's jobs, so the next job's rows are requested
    // while the current one ends.
    auto prefetch_row = [&](int ix) {
      if (ix >= 0 && ix < a.n_kv) {
        const uint8_t* r = a.kv + static_cast<size_t>(ix) * kRowBytes;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) prefetch_l2_line(r + 128 * c);
      }
    };
    int ixl = pre0;                                // index of row 32w + lane of the step
    int n1 = fetch(1), n2 = fetch(2);              // indices of steps g+1 and g+2
    // one chunk group of the step's 64 rows: wait until the MMAs of step g - 2
    // are done with it, copy, and arrive on its FULL barrier when the copies land
    auto copy_group = [&](auto grp, int g, int h) -> bool {
      constexpr int G = decltype(grp)::value;
      if (g >= 2) {
        int ok = 1;
        if (lane == 0) ok = wait_bounded(bar((G == 0 ? B_EMPTYA0 : B_EMPTYB0) + h), ((g >> 1) - 1) & 1, wc,
                                         W_PROD_EMPTY);
        if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int rl = 4 * m + ro;                   // row within the warp's 32
        const int row = 32 * warp + rl;
        const int ix = __shfl_sync(0xffffffffu, ixl, rl);
        const bool valid = ix >= 0 && ix < a.n_kv;
        const uint8_t* src = a.kv + static_cast<size_t>(valid ? ix : 0) * kRowBytes + pc * 16;
        const uint32_t dst = sbase + kOffRing + h * kHalfBytes + static_cast<uint32_t>(sw128(row, pc));
        if constexpr (G == 0) copy_row_chunks<0, kGroupSplit>(dst, src, valid ? 16u : 0u);
        else copy_row_chunks<kGroupSplit, kChunks>(dst, src, valid ? 16u : 0u);
      }
      cp_async_arrive_noinc(bar((G == 0 ? B_FULLA0 : B_FULLB0) + h));
      return true;
    };
#pragma unroll 1
    for (int g = 0; g < total; ++g) {
      const int h = g & 1;
      // (index checks on request: -1 is padding, anything else outside [0, n_kv) is reported)
      if (a.check_idx && ixl != -1 && (ixl < 0 || ixl >= a.n_kv)) atomicOr(&a.status[0], 0x10u);
      if (!copy_group(std::integral_constant<int, 0>{}, g, h) ||
          !copy_group(std::integral_constant<int, 1>{}, g, h))
        break;
      // (Deferring the first prefetches until the first two steps' copies are on
      // their way measured slower, at s_q = 1 and 96 alike.)
      if (g == 0) prefetch_row(n1);
      prefetch_row(n2);
      ixl = n1;
      n1 = n2;
      n2 = fetch(g + 3);                           // arrives while this step is computed
    }
    cp_async_wait_all();   // nothing of this thread is still landing when the CTA exits
  } else if (warp == 2) {
    // ============================================================ Q loads ===
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      int issued = 0;
#pragma unroll 1
      for (int j = 0; j < njobs; ++j) {
        const Job jb = (j == 0) ? j0 : job_at<kSched>(a, j);
        // the buffer is free once the previous job's last QK has completed; that
        // barrier has one phase per job, waited in order
        if (j > 0 && !wait_bounded(bar(B_QFREE), (j - 1) & 1, wc, W_PROD_Q)) break;
        mbar_arrive_expect_tx(bar(B_QFULL), kQBytes);
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c)
          tma_load_2d(sbase + kOffQ + c * kQChunkBytes, &tm_q, 64 * c, kMlaHeads * jb.t, bar(B_QFULL));
        ++issued;
        // the next job's Q is requested into L2 now, so its load (once this job's
        // QKs are done) does not wait for DRAM
        if (j + 1 < njobs) {
          const int tn = job_at<kSched>(a, j + 1).t;
#pragma unroll 1
          for (int c = 0; c < kChunks; ++c) tma_prefetch_2d(&tm_q, 64 * c, kMlaHeads * tn);
        }
      }
      // Nothing this thread started may still be writing shared memory when the
      // CTA exits: wait for the last Q load (each load is issued only after the
      // previous one was consumed, so it is the only one that can be in flight;
      // already landed, unless the CTA is aborting).
      if (issued > 0 && !wait_drain(bar(B_QFULL), (issued - 1) & 1, a.drain_limit_ns))
        atomicCAS(&a.status[1], 0u, W_DRAIN_Q);
    }
  } else if (warp == 3) {
    // ========================================================= MMA issuer ===
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_make(64, 64, 1, false, false);   // A (Q), B (K rows) K-major
      constexpr uint32_t kIdescPV = idesc_make(128, 64, 1, true, false);   // A (V^T) MN-major, B (P^T) K-major
      // Operand descriptors as 32-bit words. Every descriptor's high word is the
      // same (128-byte swizzle, 1024-byte atom stride); the low word holds the
      // start address (bits 0-13, address >> 4, no carry out of it below 256 KB)
      // and the leading-byte offset, so another K step, chunk, tile or ring half
      // is an add to the low word, and within a group of MMAs that add is a
      // compile-time constant. The groups are fully unrolled: tcgen05.mma is
      // issued by one thread, and every instruction between two MMAs delays the
      // next one (measured with a probe of this stream: 48-51 cycles per MMA
      // unrolled, 60-64 with the descriptors stepped in a rolled loop).
      const uint32_t w_hi = static_cast<uint32_t>(sdesc_sw128(sbase, 16, 1024) >> 32);
      const uint32_t w_k0 = static_cast<uint32_t>(sdesc_sw128(sbase + kOffRing, 16, 1024));
      const uint32_t w_v0 = static_cast<uint32_t>(sdesc_sw128(sbase + kOffRing, kSlotBytes, 1024));
      const uint32_t w_phi0 = static_cast<uint32_t>(sdesc_sw128(sbase + kOffRing + 8 * kSlotBytes, 16, 1024));
      const uint32_t w_q = static_cast<uint32_t>(sdesc_sw128(sbase + kOffQ, 16, 1024));
      const uint32_t w_plo = static_cast<uint32_t>(sdesc_sw128(sbase + kOffPlo, 16, 1024));
      constexpr uint32_t kHalfStep = kHalfBytes >> 4;
      // QK(g) over chunks C0 .. C1-1: 4 MMAs of K=16 (32 bytes of a K-major row)
      // per 64-dim chunk, all into S buffer g & 1.
      auto qk_chunks = [&](int g, auto c0, auto c1) {
        constexpr int C0 = decltype(c0)::value, C1 = decltype(c1)::value;
        const uint32_t d = tmem + kTmemS + 64 * (g & 1);
        const uint32_t bk = w_k0 + (g & 1) * kHalfStep;
#pragma unroll
        for (int c = C0; c < C1; ++c) {
          if (c == 0) mma_f16_wc<0>(d, w_q, bk, w_hi, kIdescQK);
          else mma_f16_wc<1>(d, w_q + c * (kQChunkBytes >> 4), bk + c * (kSlotBytes >> 4), w_hi, kIdescQK);
#pragma unroll
          for (int kk = 1; kk < 4; ++kk)
            mma_f16_wc<1>(d, w_q + c * (kQChunkBytes >> 4) + 2 * kk, bk + c * (kSlotBytes >> 4) + 2 * kk, w_hi,
                          kIdescQK);
        }
      };
      // This CTA's O^T tiles: tq0 .. tq0 + nq - 1 (all four unless the job's dims
      // are spread over several CTAs).
      const int tq0 = j0.q0;
      const uint32_t v_q0 = w_v0 + static_cast<uint32_t>(tq0) * ((2 * kSlotBytes) >> 4);
      const uint32_t d_q0 = tmem + 64u * static_cast<uint32_t>(tq0);
      // PV(g) for the CTA's tile J (dims 128 (tq0 + J) .. + 127) with P_hi (part 0)
      // or P_lo (part 1): K = the 64 rows in 4 steps of 16 (2048 B of the MN-major
      // V^T, 32 B of the K-major P^T each). acc0 = 0 starts a new O^T (first step
      // of a job): it is the first MMA's accumulate predicate, not a branch.
      // `par` moves tiles 0 and 1 of an odd job to their second place (tile_col).
      // Every run of MMAs is straight-line code (J is a constant once the callers'
      // loops are unrolled; conditional commits are predicated instructions): a
      // branch between two MMAs measured about as costly as another MMA.
      auto pv_tile = [&](int g, auto part, int J, uint32_t acc0, uint32_t par) {
        constexpr int kPart = decltype(part)::value;
        const uint32_t av = v_q0 + (g & 1) * kHalfStep + J * ((2 * kSlotBytes) >> 4);
        const uint32_t bp = kPart ? w_plo : w_phi0 + (g & 1) * kHalfStep;
        const uint32_t d = d_q0 + 64 * J + (J < 2 ? par : 0u);
        mma_f16_w(d, av, bp, w_hi, kIdescPV, kPart ? 1u : acc0);
        mma_f16_wc<1>(d, av + (2048 >> 4), bp + 2, w_hi, kIdescPV);
        mma_f16_wc<1>(d, av + (4096 >> 4), bp + 4, w_hi, kIdescPV);
        mma_f16_wc<1>(d, av + (6144 >> 4), bp + 6, w_hi, kIdescPV);
      };
      constexpr std::integral_constant<int, 0> kHi{};
      constexpr std::integral_constant<int, 1> kLo{};
      bool ok = true;
      auto wait = [&](uint32_t b, uint32_t ph, uint32_t site) {
        if (ok && !wait_bounded(b, ph, wc, site)) ok = false;
        return ok;
      };
      // the rows were written by other threads' cp.async (generic proxy); make
      // them visible to the tensor core's reads (async proxy)
      auto rows_visible = [&]() {
        fence_proxy_async_smem();
        tc_fence_after();
      };
      // QK(g) in its two chunk groups, each after its rows have landed; the first
      // step of a job also waits for the job's Q, the last one releases it.
      auto issue_qk = [&](int g, const Step& st) {
        const int h = g & 1;
        if (!wait(bar(B_FULLA0 + h), (g >> 1) & 1, W_MMA_STALL)) return false;
        if (st.first && !wait(bar(B_QFULL), st.job & 1, W_MMA_Q)) return false;
        rows_visible();
        qk_chunks(g, std::integral_constant<int, 0>{}, std::integral_constant<int, kGroupSplit>{});
        if (!wait(bar(B_FULLB0 + h), (g >> 1) & 1, W_MMA_STALL)) return false;
        rows_visible();
        qk_chunks(g, std::integral_constant<int, kGroupSplit>{}, std::integral_constant<int, kChunks>{});
        mma_commit(bar(B_SFULL0 + h));
        if (st.last) mma_commit(bar(B_QFREE));   // the job's QKs are all issued
        return true;
      };
      // PV(g) over the CTA's kNq tiles with the release of its chunk groups:
      // tile-major (P_hi and P_lo of a tile together, so group A frees after the
      // first two tiles) when P_lo is published already, else all P_hi tiles
      // first (P_lo's buffer is still being read by PV(g - 1) when PV(g) is
      // issued right behind it). Group A (chunks 0-3) is read by tiles 0 and 1
      // only: it is released after the last of those the CTA computes, or before
      // the run when it computes neither. On the job's last step each O^T tile's
      // completion is signalled on its own barrier (B_OT0 + tile), so the
      // epilogue reads a tile while the MMAs of the next ones still run. The
      // first step of a job after the first (kBoundary) writes tiles 2 and 3 only
      // once the epilogue of the job before has read them.
      auto issue_pv = [&](int g, const Step& st, auto tile_major, auto nq, auto boundary) {
        constexpr bool kTileMajor = decltype(tile_major)::value;
        constexpr bool kBoundary = decltype(boundary)::value;
        constexpr int kNq = decltype(nq)::value;
        constexpr int kAAfter = kNq == 4 ? 1 : kNq - 1;
        const int h = g & 1;
        const uint32_t acc0 = st.first ? 0u : 1u, lastu = st.last ? 1u : 0u;
        const uint32_t par = (st.job & 1) ? kTmemAlt : 0u;
        const uint32_t a_lead = tq0 >= 2 ? 1u : 0u;
        auto tile_free = [&](int J) {   // (kBoundary only) tile J of the previous job has been read
          if (!wait(bar(J == 2 ? B_OFREE2 : B_OFREE3), (st.job - 1) & 1, W_MMA_STALL)) return false;
          tc_fence_after();
          return true;
        };
        if (!wait(bar(B_PHI0 + h), (g >> 1) & 1, W_MMA_STALL)) return false;
        if (kTileMajor && !wait(bar(B_PLO0 + h), (g >> 1) & 1, W_MMA_STALL)) return false;
        tc_fence_after();
        mma_commit_if(bar(B_EMPTYA0 + h), a_lead);
        if constexpr (kTileMajor) {
#pragma unroll
          for (int J = 0; J < kNq; ++J) {
            if (kBoundary && J >= 2 && !tile_free(J)) return false;
            pv_tile(g, kHi, J, acc0, par);
            pv_tile(g, kLo, J, acc0, par);
            mma_commit_if(bar(B_OT0 + tq0 + J), lastu);
            if (J == kAAfter) mma_commit_if(bar(B_EMPTYA0 + h), a_lead ^ 1u);
          }
        } else {
#pragma unroll
          for (int J = 0; J < kNq; ++J) {
            if (kBoundary && J >= 2 && !tile_free(J)) return false;
            pv_tile(g, kHi, J, acc0, par);
          }
          if (!wait(bar(B_PLO0 + h), (g >> 1) & 1, W_MMA_STALL)) return false;
          tc_fence_after();
#pragma unroll
          for (int J = 0; J < kNq; ++J) {
            pv_tile(g, kLo, J, 1u, par);
            mma_commit_if(bar(B_OT0 + tq0 + J), lastu);
            if (J == kAAfter) mma_commit_if(bar(B_EMPTYA0 + h), a_lead ^ 1u);
          }
        }
        mma_commit(bar(B_EMPTYB0 + h));   // the half is free for the rows of step g + 2
        mma_commit(bar(B_PVDONE));
        return true;
      };
      // A fixed order by pairs of steps over all of the CTA's jobs,
      //   QK(g) QK(g+1) PV(g) PV(g+1),
      // each group issued after its own bounded waits. Every wait's producer was
      // issued earlier in this order (the rows of g+1 come after PV(g-1) freed
      // its half, P_lo(g) after PV(g-1) is done, S(g)'s buffer is free once
      // PV(g-2) is issued, a job's Q after the previous job's last QK, the
      // previous job's O^T tiles are read once PV of its last step is done), so
      // the order cannot deadlock. QK(g+1) covers the softmax of g, PV(g) that of
      // g+1; the chunk groups of step g's half are refilled with the rows of g+2
      // while PV(g+1) and QK(g+2) run.
      auto run = [&](auto nq) {
        constexpr int kNq = decltype(nq)::value;
        auto pv = [&](int g, const Step& st, auto tm) {
          if constexpr (kNq == 4 && kSched != 0) {
            if (st.first && st.job > 0) return issue_pv(g, st, tm, nq, std::true_type{});
          }
          return issue_pv(g, st, tm, nq, std::false_type{});
        };
#pragma unroll 1
        for (int g = 0; g < total && ok; g += 2) {
          const bool two = g + 1 < total;
          const Step s0 = step_at<kSched>(a, j0, u0, total, g);
          const Step s1 = two ? step_at<kSched>(a, j0, u0, total, g + 1) : s0;
          if (!issue_qk(g, s0)) break;
          if (two && !issue_qk(g + 1, s1)) break;
          if (!pv(g, s0, std::true_type{})) break;
          if (two && !pv(g + 1, s1, std::false_type{})) break;
        }
      };
      if (kSched != 0 || j0.nq == 4) run(std::integral_constant<int, 4>{});   // (balanced: always 4)
      else if constexpr (kSched == 0) {
        if (j0.nq == 2) run(std::integral_constant<int, 2>{});
        else run(std::integral_constant<int, 1>{});
      }
      if (!ok) {
        // no MMA may still be reading shared memory or writing TMEM when the CTA exits
        mma_commit(bar(B_DRAIN));
        if (!wait_drain(bar(B_DRAIN), 0, a.drain_limit_ns)) atomicCAS(&a.status[1], 0u, W_DRAIN_MMA);
      }
    }
  } else {
    // ============================================== softmax + epilogue ====
    const int sp = warp & 3;               // TMEM sub-partition (lanes 32sp..32sp+31)
    const uint32_t lane_base = static_cast<uint32_t>(32 * sp) << 16;
    const int head = 16 * sp + (lane & 15);   // this thread's head
    const int rb = (lane >> 4) * 32;          // and its 32 rows rb..rb+31 of every step
    int bad = 0;               // a bounded wait of this warp ran out
    float amax_l = 0.f;        // max |O| over the final rows this thread wrote
    auto bounded = [&](uint32_t b, uint32_t ph, uint32_t site) {
      int w = 1;
      if (lane == 0) w = wait_bounded(b, ph, wc, site);
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) bad = 1;
      return w != 0;
    };

    // The end of job jj: the softmax denominator and the job's own LSE per head
    // into hs[jj & 1] (1/denominator, LSE), and the LSE to global memory.
    auto finalize = [&](const Job& J, int jj, float m_run, float lsum) {
      lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
      const float lse_own = lsum > 0.f ? m_run + log2f(lsum) : -INFINITY;
      if (lane < 16) {
        float den = lsum;
        if (J.kind == J_FINAL && a.sink != nullptr && lsum > 0.f) den += exp2f(a.sink[head] * kLog2e - m_run);
        float* hj = hs + (jj & 1) * 128;
        hj[head] = lsum > 0.f ? 1.f / den : 0.f;
        hj[64 + head] = lse_own;
        if (!bad && J.q0 == 0) {   // (every CTA of a job has the same LSE)
          if (J.kind == J_FINAL) {
            if (a.lse_out != nullptr) a.lse_out[J.out_row + head] = lse_own;
          } else {
            a.lse_acc[J.out_row + head] = lse_own;
          }
        }
      }
    };
    // The epilogue of job J (the CTA's job jj), straight from TMEM to global
    // memory. O^T tile q holds dims 128q .. 128q+127 in its lanes and the 64
    // heads in its columns: this thread handles dim d of every head; for each
    // head the warp's 32 lanes touch 32 consecutive dims. `deferred` (balanced
    // schedule): the next job has started, and its first PV waits for tiles 2
    // and 3 (taken first, each released right after its read); tiles 0 and 1 of
    // the next job have their own place.
    auto epilogue = [&](const Job& J, int jj, bool deferred) {
      const float* hj = hs + (jj & 1) * 128;
#pragma unroll 1
      for (int i = 0; i < J.nq; ++i) {
        const int q = deferred ? ((i + 2) & 3) : J.q0 + i;
        const int d = 128 * q + 32 * sp + lane;
        // Deferred, tiles 0 and 1 are not waited for: the commits of tiles 2 and
        // 3, waited first, track every earlier MMA of the job; and the next
        // job's first PV, free to write its own tiles 0 and 1, may already have
        // completed their barriers' next phase (a one-step job), which a wait
        // on this job's phase would then take for the one after.
        if (!bad && (!deferred || q >= 2)) bounded(bar(B_OT0 + q), jj & 1, W_SM_PV_EPI);
        tc_fence_after();
        float v[64];
        {
          uint32_t o[64];
          tmem_ld_32x32b_x64(tmem + lane_base + tile_col(q, jj), o);
          tmem_wait_ld_x64(o);
          // the per-head factor read into registers before any store below
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            const float4 fv = *reinterpret_cast<const float4*>(hj + c);
            v[c] = __uint_as_float(o[c]) * fv.x;
            v[c + 1] = __uint_as_float(o[c + 1]) * fv.y;
            v[c + 2] = __uint_as_float(o[c + 2]) * fv.z;
            v[c + 3] = __uint_as_float(o[c + 3]) * fv.w;
          }
        }
        if (kSched != 0 && q >= 2) {
          // this warp's read of the tile is done: the next job's first PV may write it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(q == 2 ? B_OFREE2 : B_OFREE3));
        }
        if (J.kind == J_FINAL) {
          amax_l = fmaxf(amax_l, store_final(a, J.t, d - lane, lane, v));
        } else if (a.partial_bf16) {
          // bf16 partials: the rows of the final bf16 output's layout, at the slot
          store_rows(reinterpret_cast<__nv_bfloat16*>(a.o_acc) + J.out_row * kMlaDv, 1, 1.f, d - lane, lane, v);
        } else {
          float* st = a.o_acc + J.out_row * kMlaDv + d;
#pragma unroll
          for (int c = 0; c < 64; ++c) st[c * kMlaDv] = v[c];
        }
      }
    };

    Job jb = j0;               // the job of the current step
    int job = 0;
    Job jp = j0;               // a finished job whose epilogue is still to run
    int pend = -1;
    float m_run = -INFINITY;   // reference max of the head (log2 units), shared by its two lanes
    float lsum = 0.f;          // fp32 softmax denominator over this thread's rows
    int ia = pre0, ib = pre1;  // indices of rows lane and lane + 32 of the step
    int g = 0;
#pragma unroll 1
    for (; g < total && !bad; ++g) {
      const int h = g & 1;
      const Step st = step_at<kSched>(a, j0, u0, total, g);
      if (st.first && g > 0) {
        job = st.job;
        jb = job_at<kSched>(a, job);
        m_run = -INFINITY;
        lsum = 0.f;
      }
      // which of this thread's 32 rows hold a valid index
      const uint32_t vlo = __ballot_sync(0xffffffffu, ia >= 0 && ia < a.n_kv);
      const uint32_t vhi = __ballot_sync(0xffffffffu, ib >= 0 && ib < a.n_kv);
      const uint32_t vm = rb ? vhi : vlo;
      if (g + 1 < total) {   // the next step's indices, in flight during this step
        const Step sn = step_at<kSched>(a, j0, u0, total, g + 1);
        const int32_t* idx_n = a.idx + static_cast<size_t>(sn.t) * a.topk;
        const int rn = sn.r0 + lane;
        ia = rn < sn.r1 ? __ldg(idx_n + rn) : -1;
        ib = rn + 32 < sn.r1 ? __ldg(idx_n + rn + 32) : -1;
      }

      const bool w = bounded(bar(B_SFULL0 + h), (g >> 1) & 1, W_SM_S);
      tc_fence_after();
      float x[32];
      float mx = -INFINITY;
      if (w) {
        uint32_t raw[32];
        tmem_ld_16x32bx2_x32_h32(tmem + lane_base + kTmemS + 64 * h, raw);
        tmem_wait_ld_x32(raw);
        if (vm == 0xffffffffu) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            x[i] = __uint_as_float(raw[i]) * a.scale_log2;
            mx = fmaxf(mx, x[i]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            x[i] = ((vm >> i) & 1u) ? __uint_as_float(raw[i]) * a.scale_log2 : -INFINITY;
            mx = fmaxf(mx, x[i]);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = -INFINITY;
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));   // over the step's 64 rows

      // Lazy rescale: move the reference max only when a score exceeds it by
      // more than the threshold (always on the first valid row of a head). Both
      // lanes of the head see the same mx and take the same decision.
      const bool need = mx > m_run + kRescaleThreshold;
      if (need) {
        const float al = (m_run == -INFINITY) ? 0.f : ex2_approx(m_run - mx);
        lsum *= al;
        m_run = mx;
        if (lane < 16) alpha_s[h * 64 + head] = al;
      }
      const uint32_t rmask = __ballot_sync(0xffffffffu, need) & 0xffffu;
      __syncwarp();
      if (lane == 0) {
        xch[h * 4 + sp] = rmask | (bad ? 0x10000u : 0u);
        mbar_arrive(bar(B_XCH0 + h));      // release: the mask and the factors above
      }

      // p = 2^(x - m_ref); a masked row gives 0
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = (x[i] == -INFINITY) ? 0.f : ex2_approx(x[i] - m_run);
      {
        float ts[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) ts[i] = x[i] + x[i + 16];
#pragma unroll
        for (int i = 0; i < 8; ++i) ts[i] += ts[i + 8];
#pragma unroll
        for (int i = 0; i < 4; ++i) ts[i] += ts[i + 4];
        lsum += (ts[0] + ts[2]) + (ts[1] + ts[3]);
      }
      // P_hi = p with its mantissa cut to bf16 (exact bit truncation, no
      // conversion); P_lo = bf16(p - P_hi), two rows per packed conversion.
      // |P_lo| < 2^-7 p, so P_hi + P_lo matches p to 2^-15.
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const uint32_t b0 = __float_as_uint(x[i]) & 0xFFFF0000u;
        const uint32_t b1 = __float_as_uint(x[i + 1]) & 0xFFFF0000u;
        const __nv_bfloat162 lo2 =
            __floats2bfloat162_rn(x[i] - __uint_as_float(b0), x[i + 1] - __uint_as_float(b1));
        hi[i / 2] = (b0 >> 16) | b1;
        lo[i / 2] = *reinterpret_cast<const uint32_t*>(&lo2);
      }

      // The other warps' rescale masks for this step.
      const bool wx = bounded(bar(B_XCH0 + h), (g >> 1) & 1, W_SM_X);
      const uint32_t x0 = xch[h * 4 + 0], x1 = xch[h * 4 + 1], x2 = xch[h * 4 + 2], x3 = xch[h * 4 + 3];
      if (((x0 | x1 | x2 | x3) & 0x10000u) || !wx) {
        bad = 1;
        break;   // every softmax warp sees the same masks and leaves together
      }
      const uint64_t resc = static_cast<uint64_t>(x0) | (static_cast<uint64_t>(x1) << 16) |
                            (static_cast<uint64_t>(x2) << 32) | (static_cast<uint64_t>(x3) << 48);
      // P^T as a K-major operand: N = heads, K = rows; the 64 rows of one head
      // are one 128-byte line of the swizzled tile, this thread's 32 rows are
      // its pieces rb/8 .. rb/8+3.
      uint8_t* p_hi = smem + kOffRing + 8 * kSlotBytes + h * kHalfBytes;
      uint8_t* p_lo = smem + kOffPlo;
      auto store_p = [&](uint8_t* dst, const uint32_t (&v)[16]) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(dst + sw128(head, (rb >> 3) + q)) =
              make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      };
      auto publish = [&](int b) {   // generic-proxy stores -> the tensor core's reads
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(b));
      };
      if (resc == 0 || st.first) {
        // O^T needs no rescale before PV_hi(g) (or holds nothing of this job
        // yet): publish P_hi now; P_lo's buffer is free once PV(g-1) is done.
        store_p(p_hi, hi);
        publish(B_PHI0 + h);
        if (g >= 1) {
          bounded(bar(B_PVDONE), (g - 1) & 1, W_SM_PV);
          tc_fence_after();
        }
        store_p(p_lo, lo);
        publish(B_PLO0 + h);
      } else {
        // O^T holds PV of this job's earlier steps: once PV(g-1) is done, scale
        // the columns of the rescaled heads in the 32 dims (TMEM lanes) of each
        // tile this warp can reach, then publish both halves of P.
        bounded(bar(B_PVDONE), (g - 1) & 1, W_SM_PV);
        tc_fence_after();
        if (!bad) {
#pragma unroll 1
          for (int q = 2 * jb.q0; q < 2 * (jb.q0 + jb.nq); ++q) {   // own O^T tiles x 2 halves of 32 heads
            const int c0 = 32 * (q & 1);
            if (((resc >> c0) & 0xffffffffull) == 0) continue;
            uint32_t o[32];
            float al[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) al[i] = ((resc >> (c0 + i)) & 1ull) ? alpha_s[h * 64 + c0 + i] : 1.f;
            const uint32_t col = tile_col(q >> 1, job) + c0;
            tmem_ld_32x32b_x32(tmem + lane_base + col, o);
            tmem_wait_ld_x32(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * al[i]);
            tmem_st_32x32b_x32(tmem + lane_base + col, o);
          }
          tmem_wait_st();
        }
        store_p(p_hi, hi);
        store_p(p_lo, lo);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(B_PHI0 + h));
          mbar_arrive(bar(B_PLO0 + h));
        }
      }

      // The previous job's epilogue, now that this (its successor's first) step
      // is published: the issuer computes this job's first PV meanwhile.
      if (kSched != 0) {
        if (pend >= 0) {
          epilogue(jp, pend, true);
          pend = -1;
        }
        if (st.last) {
          finalize(jb, job, m_run, lsum);
          if (g + 1 < total) {
            jp = jb;
            pend = job;
          }
        }
      }
    }

    if (kSched == 0 && !bad) finalize(jb, job, m_run, lsum);   // (the one job of the uniform schedule)
    // ---- epilogue of the last job -------------------------------------------
    // Every softmax warp reaches this named barrier (a failed wait only ends the
    // step loop after the exchange that follows it), so none can wait there
    // forever; it also makes every warp's per-head scalars visible.
    if (lane == 0) fin[sp] = bad;
    named_bar_sync(1, 128);
    if (fin[0] | fin[1] | fin[2] | fin[3]) bad = 1;
    if (!bad) epilogue(jb, job, false);
    if (a.amax != nullptr && !bad) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax_l = fmaxf(amax_l, __shfl_xor_sync(0xffffffffu, amax_l, o));
      if (lane == 0 && amax_l > 0.f) atomicMax(reinterpret_cast<int*>(a.amax), __float_as_int(amax_l));
    }
  }

  // ---- teardown: every role reaches this point, TMEM is freed by its owner --
  tc_fence_before();
  __syncthreads();
  if (warp == 3) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int mla_decode_smem_bytes() { return kSmemBytes; }

cudaError_t prepare_mla_kernels() {
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  const cudaError_t e =
      cudaFuncSetAttribute(mla_decode_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mla_decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_mla_decode(const CUtensorMap& tm_q, const MlaArgs& a, cudaStream_t stream) {
  if (a.sched == 0 && a.dim_groups != 1 && a.dim_groups != 2 && a.dim_groups != 4) return cudaErrorInvalidValue;
  if (a.sched == 0 && a.tail_splits > 0 && (a.num_splits != 1 || a.dim_groups != 1 || a.tail_first < 0 ||
                                            a.tail_first >= a.s_q || a.tail_dgroups != 0))
    return cudaErrorInvalidValue;
  if (a.sched == 0 && a.tail_dgroups != 0 &&
      ((a.tail_dgroups != 2 && a.tail_dgroups != 4) || a.num_splits != 1 || a.dim_groups != 1 ||
       a.tail_first < 0 || a.tail_first >= a.s_q || !a.direct_whole))
    return cudaErrorInvalidValue;
  const int tail_per = a.tail_splits > 0 ? a.tail_splits : a.tail_dgroups;   // CTAs per tail token
  const dim3 grid(a.sched != 0 ? static_cast<unsigned>(a.num_ctas)
                  : tail_per > 0
                      ? static_cast<unsigned>(a.tail_first) +
                            static_cast<unsigned>(a.s_q - a.tail_first) * static_cast<unsigned>(tail_per)
                      : static_cast<unsigned>(a.s_q) * static_cast<unsigned>(a.num_splits) *
                            static_cast<unsigned>(a.dim_groups));
  // launched as a programmatic dependent of the preceding kernel on the stream:
  // its CTAs may become resident and set up while that kernel finishes
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.sched == 0) return cudaLaunchKernelEx(&cfg, mla_decode_kernel<0>, tm_q, a);
  return cudaLaunchKernelEx(&cfg, mla_decode_kernel<1>, tm_q, a);
}

// ---- bounded-wait self test ---------------------------------------------------

__global__ void wait_selftest_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t b;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&b), 1);
    abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtx wc{limit_ns, status, &abort_flag};
    (void)wait_bounded(smem_u32(&b), 0, wc, 0x5E1F);   // nothing ever arrives
  }
}

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace skv

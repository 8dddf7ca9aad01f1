// Dense split-KV FP8 SDPA decode for sm_103a (the form of cuDNN-frontend PR #768,
// SM120 FP8 commit): per-tensor scaled e4m3 Q/K/V, GQA, bottom-right causal
// mask, the KV range of each sequence cut into near-equal runs of 128-key
// tiles with the remainder to the leading splits, fp32 partial O + log2 LSE
// into split-major slots (or, unsplit, a direct bf16/fp32/e4m3 epilogue that
// also computes the amax).
//
// One CTA per job (sequence b, KV head g, split s), 448 threads:
//   warp 0     TMA: the job's Q rows once (the group's h_q/h_kv heads of up to
//              64/group tokens = 64 rows x 128 B), then per tile K and V
//              (128 keys x 128 B each, e4m3) into a 3-stage ring.
//   warp 1     tcgen05 issue:  S[64 rows x 128 keys] = Q . K^T     (kind::f8f6f4, K=128)
//                              O^T[128 d x 64 rows] += V^T . P^T   (kind::f16, f16 operands)
//   warps 2-9  softmax over the keys of each query row (S = Q.K^T, M=64: two
//              warps per TMEM sub-partition, each with 64 of the tile's 128 keys,
//              32 per thread), lazy rescale of O^T, P^T in f16, then the epilogue.
//   warps 10-13 convert each V tile from e4m3 to f16 (exact) into the
//              MN-major 128-byte-swizzled layout the PV MMA reads.
// The QK product of e4m3 codes is exact in fp32; descales multiply the scores
// (dq*dk*sm_scale) and the output (dv).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"
#include "softmax_util.cuh"

namespace skv {
namespace {

// Four e4m3 codes (bytes 0..3 of w) to four f16 values, exactly (every e4m3
// value, subnormals included, is an f16 value; the NaN codes stay NaN), with the
// hardware's paired conversion: bytes 0, 1 -> lo, bytes 2, 3 -> hi, low half
// first. (An integer form that places the code's bits inside an f16, reading its
// value times 2^-8, takes four integer operations per pair; on this kernel's
// busiest pipe that measured ~8 % slower.)
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const __half2_raw a = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFFu), __NV_E4M3);
  const __half2_raw b = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
  lo = *reinterpret_cast<const uint32_t*>(&a);
  hi = *reinterpret_cast<const uint32_t*>(&b);
}

constexpr int kKeyWarps = 2;              // softmax warps per TMEM sub-partition, splitting a tile's keys
constexpr int kSoftmaxWarps = 4 * kKeyWarps;   // warps 2 .. 1 + kSoftmaxWarps
constexpr int kKPT = 64 / kKeyWarps;       // keys of a tile per softmax thread
constexpr int kCPW = 64 / kKeyWarps;       // O^T columns (query rows) per softmax warp in the epilogue
constexpr int kConverters = 4;             // the last 4 warps: one key row of the V tile per thread
constexpr int kFirstConverter = 2 + kSoftmaxWarps;
constexpr int kThreads = 32 * (kFirstConverter + kConverters);
static_assert(kKeyWarps == 2, "the TMEM load shapes and the 32-score max below");
constexpr int kD = 128;
constexpr int kTile = 128;                 // keys per tile (split unit)
constexpr int kRows = 64;                  // query rows per job (tokens x group heads)
constexpr int kStages = 3;
constexpr int kKVTileBytes = kTile * kD;   // 16384 (e4m3)
constexpr int kStageBytes = 2 * kKVTileBytes;
constexpr int kV16Bytes = kTile * kD * 2;  // 32768
constexpr int kPBytes = kRows * kTile * 2; // 16384
constexpr int kQBytes = kRows * kD;        // 8192

constexpr int kOffStage = 0;
constexpr int kOffV16 = kOffStage + kStages * kStageBytes;   // 98304
constexpr int kOffP = kOffV16 + 2 * kV16Bytes;               // 163840
constexpr int kPBuffers = 3;               // P(t) in buffer t % 3 (see the MMA loop)
constexpr int kOffQ = kOffP + kPBuffers * kPBytes;           // 212992
constexpr int kOffBars = kOffQ + kQBytes;                    // 221184
constexpr int kOffMisc = kOffBars + 256;
constexpr int kOffAlpha = kOffMisc + 128;                    // float[2][64] rescale factors by tile parity
constexpr int kOffInv = kOffAlpha + 512;                     // float[64] dv / l per row
constexpr int kOffHalf = kOffInv + 256;                      // float[2][kKeyWarps][64] per-row maxima of each
                                                             // key part by tile parity, then float[kKeyWarps][64]
                                                             // row sums
constexpr int kOffFlags = kOffHalf + 3 * kKeyWarps * 256;    // int[2][kSoftmaxWarps] per-tile words, int[kSoftmaxWarps]
constexpr int kSmemUsed = kOffFlags + 3 * kSoftmaxWarps * 4;
constexpr int kSmemBytes = kSmemUsed + 1024;

enum {
  B_QFULL = 0, B_SFULL_STAGE0, B_SFULL_STAGE1, B_SFULL_STAGE2, B_SEMPTY0, B_SEMPTY1, B_SEMPTY2,
  B_SREADY0, B_SREADY1, B_PFULL0, B_PFULL1, B_V16FULL0, B_V16FULL1, B_V16EMPTY0, B_V16EMPTY1,
  B_FINAL, B_DRAIN, B_PVDONE, kNumBars
};
static_assert(kNumBars * 8 <= 256, "barrier area");

constexpr uint32_t kTmemCols = 512;        // O^T at [0, 64), S buffers (128 keys each) at 128 and 256
constexpr uint32_t kTmemS = 128;
constexpr float kRescaleThreshold = 8.0f;

enum : uint32_t {
  W_PROD = 101, W_MMA_Q, W_MMA_P, W_MMA_V, W_MMA_FULL, W_SM_S, W_SM_FINAL, W_CV_FULL, W_CV_EMPTY,
  W_DRAIN_MMA2, W_DRAIN_TMA2, W_SM_PV
};

// TMEM moves chosen by the register count (the softmax warps' share of a tile
// or of O^T depends on how many warps split it).
template <int N>
__device__ __forceinline__ void tld_16x32bx2_h32(uint32_t a, uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "shape");
  if constexpr (N == 32) tmem_ld_16x32bx2_x32_h32(a, r);
  else tmem_ld_16x32bx2_x16_h32(a, r);
}
template <int N>
__device__ __forceinline__ void tld_32x32b(uint32_t a, uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "shape");
  if constexpr (N == 32) tmem_ld_32x32b_x32(a, r);
  else tmem_ld_32x32b_x16(a, r);
}
template <int N>
__device__ __forceinline__ void tst_32x32b(uint32_t a, const uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "shape");
  if constexpr (N == 32) tmem_st_32x32b_x32(a, r);
  else tmem_st_32x32b_x16(a, r);
}
template <int N>
__device__ __forceinline__ void twait_ld(uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "shape");
  if constexpr (N == 32) tmem_wait_ld_x32(r);
  else tmem_wait_ld_x16(r);
}

__global__ void __launch_bounds__(kThreads, 1)
    sdpa_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const SdpaArgs a, const int direct) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Launched as a programmatic dependent: the CTA may be resident before the
  // preceding kernel on the stream is done, and the job decode below already
  // reads inputs (the sequence lengths), so it waits first.
  grid_dependency_wait();

  // ---- job decode (shared by every role) ------------------------------------
  const int S = a.num_splits;   // splits per sequence (adaptive: the most any sequence gets)
  int b = 0, g = 0, s = 0, Sb = S;
  if (!a.adaptive) {
    s = blockIdx.x % S;
    const int bg = blockIdx.x / S;
    g = bg % a.h_kv;
    b = bg / a.h_kv;
  } else {
    // Sequence bb gets clamp(ceil(tiles / T), 1, S) near-equal splits, with T
    // the fewest tiles per split for which the batch's jobs (x KV heads) fit one
    // wave of num_sms CTAs (or every sequence has one split). Jobs are listed
    // sequence by sequence, (split, KV head) within one; a CTA past the last job
    // has nothing to do.
    int total = 0, longest = 1;
    for (int bb = 0; bb < a.batch; ++bb) {
      const int tb = (__ldg(a.cu_kv + bb + 1) - __ldg(a.cu_kv + bb) + kTile - 1) / kTile;
      total += tb;
      longest = max(longest, tb);
    }
    auto jobs = [&](int tt) {
      int n = 0;
      for (int bb = 0; bb < a.batch; ++bb) {
        const int tb = (__ldg(a.cu_kv + bb + 1) - __ldg(a.cu_kv + bb) + kTile - 1) / kTile;
        n += min(S, max(1, (tb + tt - 1) / tt));
      }
      return n * a.h_kv;
    };
    int T = max(1, (total * a.h_kv + a.num_sms - 1) / a.num_sms);
    while (T < longest && jobs(T) > a.num_sms) ++T;
    int j = blockIdx.x;
    b = -1;
    for (int bb = 0; bb < a.batch; ++bb) {
      const int tb = (__ldg(a.cu_kv + bb + 1) - __ldg(a.cu_kv + bb) + kTile - 1) / kTile;
      const int sb = min(S, max(1, (tb + T - 1) / T));
      if (j < sb * a.h_kv) {
        b = bb;
        Sb = sb;
        s = j / a.h_kv;
        g = j - s * a.h_kv;
        break;
      }
      j -= sb * a.h_kv;
    }
    if (b < 0) {
      grid_launch_dependents();
      return;
    }
  }
  const int group = a.h_q / a.h_kv;
  const int q0 = a.cu_q[b];
  const int sq = a.cu_q[b + 1] - q0;
  const int k0 = a.cu_kv[b];
  const int kvlen = a.cu_kv[b + 1] - k0;
  const int R = sq * group;                              // valid rows, <= 64
  const int ntiles_all = (kvlen + kTile - 1) / kTile;
  const int base = ntiles_all / Sb, rem = ntiles_all - base * Sb;
  const int tile0 = s * base + min(s, rem);
  const int nt = base + (s < rem ? 1 : 0);
  const int key_end = min((tile0 + nt) * kTile, kvlen);  // exclusive, sequence-relative
  const float dq = a.descale_q ? *a.descale_q : 1.f;
  const float dk = a.descale_k ? *a.descale_k : 1.f;
  const float dv = a.descale_v ? *a.descale_v : 1.f;
  // output row of (row rho): token q0 + rho / group, head g*group + rho % group
  auto out_index = [&](int rho) -> size_t {
    const size_t tok = static_cast<size_t>(q0 + rho / group);
    const size_t head = static_cast<size_t>(g * group + rho % group);
    return direct ? tok * a.h_q + head : (static_cast<size_t>(s) * a.total_q + tok) * a.h_q + head;
  };

  if (R > kRows) {   // more query rows than one job holds: refuse, report, write nothing
    grid_launch_dependents();
    if (threadIdx.x == 0) atomicOr(&a.status[0], 2u);
    return;
  }
  if (a.adaptive && s == 0 && !direct) {
    // the splits this sequence does not use: LSE = -inf, so the combine gives
    // them weight 0 and never reads their O
    for (int i = threadIdx.x; i < R * (S - Sb); i += kThreads) {
      const int rho = i % R, sp = Sb + i / R;
      const size_t tok = static_cast<size_t>(q0 + rho / group);
      const size_t head = static_cast<size_t>(g * group + rho % group);
      a.lse_acc[(static_cast<size_t>(sp) * a.total_q + tok) * a.h_q + head] = -INFINITY;
    }
  }
  if (nt == 0 || R <= 0) {
    // nothing to attend in this split: O = 0, LSE = -inf for the job's rows
    grid_launch_dependents();
    for (int i = threadIdx.x; i < R * kD; i += kThreads) {
      const size_t oi = out_index(i / kD) * kD + (i % kD);
      if (!direct) a.o_acc[oi] = 0.f;
      else if (a.out_dtype == 0) static_cast<float*>(a.out)[oi] = 0.f;
      else if (a.out_dtype == 1) static_cast<__nv_bfloat16*>(a.out)[oi] = __float2bfloat16_rn(0.f);
      else static_cast<uint8_t*>(a.out)[oi] = 0;
    }
    for (int i = threadIdx.x; i < R; i += kThreads) {
      if (!direct) a.lse_acc[out_index(i)] = -INFINITY;
      else if (a.lse_out != nullptr) a.lse_out[out_index(i)] = -INFINITY;
    }
    return;
  }

  auto bar = [&](int i) -> uint32_t { return sbase + kOffBars + 8 * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
  float* inv_s = reinterpret_cast<float*>(smem + kOffInv);
  const WaitCtx wc{a.wait_limit_ns, a.status, abort_flag};

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(B_SFULL_STAGE0 + i), 1);
      mbar_init(bar(B_SEMPTY0 + i), 1 + kConverters);   // QK commit + the converter warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_SREADY0 + i), 1);
      mbar_init(bar(B_PFULL0 + i), kSoftmaxWarps);
      mbar_init(bar(B_V16FULL0 + i), kConverters);
      mbar_init(bar(B_V16EMPTY0 + i), 1);
    }
    mbar_init(bar(B_FINAL), 1);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_PVDONE), 1);             // one phase per tile's PV
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(misc), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  grid_launch_dependents();   // the combine may start launching; it waits for this grid

  if (warp == 0) {
    // ======================================================= TMA producer ===
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(B_QFULL), kQBytes);
      tma_load_3d(sbase + kOffQ, &tm_q, 0, g * group, q0, bar(B_QFULL));
      int last[kStages] = {-1, -1, -1};
#pragma unroll 1
      for (int t = 0; t < nt; ++t) {
        const int st = t % kStages;
        if (t >= kStages && !wait_bounded(bar(B_SEMPTY0 + st), ((t / kStages) - 1) & 1, wc, W_PROD)) break;
        const uint32_t dst = sbase + kOffStage + st * kStageBytes;
        mbar_arrive_expect_tx(bar(B_SFULL_STAGE0 + st), kStageBytes);
        const int key = k0 + (tile0 + t) * kTile;
        tma_load_3d(dst, &tm_k, 0, g, key, bar(B_SFULL_STAGE0 + st));
        tma_load_3d(dst + kKVTileBytes, &tm_v, 0, g, key, bar(B_SFULL_STAGE0 + st));
        last[st] = t;
      }
      // Nothing this thread started may still be writing shared memory when the
      // CTA exits: wait for the last load of every stage and for Q (all landed
      // already, unless the CTA is aborting).
      for (int st = 0; st < kStages; ++st)
        if (last[st] >= 0 && !wait_drain(bar(B_SFULL_STAGE0 + st), (last[st] / kStages) & 1, a.drain_limit_ns))
          atomicCAS(&a.status[1], 0u, W_DRAIN_TMA2);
      if (!wait_drain(bar(B_QFULL), 0, a.drain_limit_ns)) atomicCAS(&a.status[1], 0u, W_DRAIN_TMA2);
    }
  } else if (warp == 1) {
    // ========================================================= MMA issuer ===
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_make(64, 128, 0, false, false);   // e4m3 x e4m3, M=64 rows, N=128 keys
      constexpr uint32_t kIdescPV = idesc_make(128, 64, 0, true, false);    // f16, A MN-major
      // Operand descriptors as 32-bit words: every operand here is 128-byte
      // swizzled with a 1024-byte atom stride, so all share one high word, and
      // another stage, buffer or K step is an add to the low word (start address
      // >> 4, below 256 KB), a compile-time constant inside a run of MMAs. Each
      // run is straight-line code; the first PV's accumulate flag is a predicate.
      const uint32_t w_hi = static_cast<uint32_t>(sdesc_sw128(sbase, 16, 1024) >> 32);
      const uint32_t w_q = static_cast<uint32_t>(sdesc_sw128(sbase + kOffQ, 16, 1024));
      const uint32_t w_k0 = static_cast<uint32_t>(sdesc_sw128(sbase + kOffStage, 16, 1024));
      const uint32_t w_v0 = static_cast<uint32_t>(sdesc_sw128(sbase + kOffV16, 16384, 1024));
      const uint32_t w_p0 = static_cast<uint32_t>(sdesc_sw128(sbase + kOffP, 16, 1024));
      auto issue_qk = [&](int t) {
        // A = Q (64 rows x 128 B), B = the K tile (128 keys x 128 B), both K-major;
        // K = 32 e4m3 codes (32 bytes) per MMA
        const uint32_t bk = w_k0 + static_cast<uint32_t>(t % kStages) * (kStageBytes >> 4);
        const uint32_t d = tmem + kTmemS + 128 * (t & 1);
        mma_f8_wc<0>(d, w_q, bk, w_hi, kIdescQK);
        mma_f8_wc<1>(d, w_q + 2, bk + 2, w_hi, kIdescQK);
        mma_f8_wc<1>(d, w_q + 4, bk + 4, w_hi, kIdescQK);
        mma_f8_wc<1>(d, w_q + 6, bk + 6, w_hi, kIdescQK);
      };
      auto issue_pv = [&](int t) {
        // A = V^T (MN-major f16, 2048 B per 16 keys), B = P^T (K-major f16, 32 B
        // per 16 keys within each 64-key atom of 8192 B)
        const uint32_t av = w_v0 + static_cast<uint32_t>(t & 1) * (kV16Bytes >> 4);
        const uint32_t bp = w_p0 + static_cast<uint32_t>(t % kPBuffers) * (kPBytes >> 4);
        mma_f16_w(tmem, av, bp, w_hi, kIdescPV, t > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 1; kk < 8; ++kk)
          mma_f16_wc<1>(tmem, av + kk * (2048 >> 4), bp + (kk >> 2) * (8192 >> 4) + (kk & 3) * 2, w_hi, kIdescPV);
      };
      // Iteration u: QK(u) as soon as its K tile has landed and its S buffer is
      // free (softmax(u-2), the buffer's last reader, has published P(u-2)), then
      // PV(u-2). The scores of tile u depend only on P(u-2), not on PV(u-2) or
      // PV(u-1), so they are ready while the softmax still works on tile u-1 (with
      // PV(t-1) issued before QK(t+1), the softmax waited ~0.3 us for its scores
      // every tile). PV runs two tiles behind, within its V16 double buffer; P has
      // three buffers: softmax(u) writes buffer u % 3 once S(u) is ready, and that
      // buffer's last reader, PV(u-3), was issued before QK(u), so it is done.
      auto pv_step = [&](int u) {
        const bool w = wait_bounded(bar(B_PFULL0 + (u & 1)), (u >> 1) & 1, wc, W_MMA_P) &&
                       wait_bounded(bar(B_V16FULL0 + (u & 1)), (u >> 1) & 1, wc, W_MMA_V);
        if (w) {
          tc_fence_after();
          issue_pv(u);
          mma_commit(bar(B_V16EMPTY0 + (u & 1)));
          mma_commit(bar(B_PVDONE));
        }
        return w;
      };
      bool ok = wait_bounded(bar(B_QFULL), 0, wc, W_MMA_Q);
#pragma unroll 1
      for (int u = 0; ok && u < nt + 2; ++u) {
        if (u < nt) {
          if (u >= 2 && !(ok = wait_bounded(bar(B_PFULL0 + (u & 1)), ((u - 2) >> 1) & 1, wc, W_MMA_P))) break;
          if (!(ok = wait_bounded(bar(B_SFULL_STAGE0 + u % kStages), (u / kStages) & 1, wc, W_MMA_FULL))) break;
          tc_fence_after();
          issue_qk(u);
          mma_commit(bar(B_SREADY0 + (u & 1)));
          mma_commit(bar(B_SEMPTY0 + u % kStages));
        }
        if (u >= 2) ok = pv_step(u - 2);
      }
      if (ok) mma_commit(bar(B_FINAL));
      if (!ok) {
        mma_commit(bar(B_DRAIN));
        if (!wait_drain(bar(B_DRAIN), 0, a.drain_limit_ns)) atomicCAS(&a.status[1], 0u, W_DRAIN_MMA2);
      }
    }
  } else if (warp >= kFirstConverter) {
    // ==================================================== V e4m3 -> f16 ===
    const int key = threadIdx.x - 32 * kFirstConverter;   // 0..127: this thread's key row of each tile
    const int r8 = key & 7;
#pragma unroll 1
    for (int t = 0; t < nt; ++t) {
      const int st = t % kStages;
      int w = 1;
      if (lane == 0) {
        w = wait_bounded(bar(B_SFULL_STAGE0 + st), (t / kStages) & 1, wc, W_CV_FULL);
        if (w && t >= 2) w = wait_bounded(bar(B_V16EMPTY0 + (t & 1)), ((t - 2) >> 1) & 1, wc, W_CV_EMPTY);
      }
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) break;   // the abort flag is set; the other roles stop on their own waits
      {
        const uint8_t* vrow = smem + kOffStage + st * kStageBytes + kKVTileBytes + (key >> 3) * 1024 + r8 * 128;
        uint8_t* v16 = smem + kOffV16 + (t & 1) * kV16Bytes + (key >> 3) * 1024 + r8 * 128;
        uint4 row[8];   // the whole 128-byte row first: eight loads in flight
#pragma unroll
        for (int c = 0; c < 8; ++c) row[c] = *reinterpret_cast<const uint4*>(vrow + ((c ^ r8) << 4));
#pragma unroll
        for (int c = 0; c < 8; ++c) {            // 16 e4m3 values (d = 16c .. 16c+15) per chunk
          const uint4 raw = row[c];
          const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t h[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) e4m3x4_to_f16x4(wds[j], h[2 * j], h[2 * j + 1]);
          // d = 16c .. 16c+7 -> MN atom (16c)/64, 16-B chunk ((16c)%64)/8; then +8
          const int d0 = 16 * c;
          const int a0 = d0 >> 6, c0 = (d0 & 63) >> 3;
          *reinterpret_cast<uint4*>(v16 + a0 * 16384 + ((c0 ^ r8) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(v16 + a0 * 16384 + (((c0 + 1) ^ r8) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_V16FULL0 + (t & 1)));
        mbar_arrive(bar(B_SEMPTY0 + st));
      }
    }
  } else {
    // ============================================== softmax + epilogue ====
    // S = Q.K^T is an M=64 accumulator: row r (token r / group, head r % group)
    // sits in lane r % 16 of sub-partition r / 16, the tile's 128 keys in its
    // columns. kKeyWarps warps share each sub-partition and split the keys:
    // warp kw of sub-partition sp reads columns c0 .. c0 + kKPT - 1 with its
    // lanes 0-15 and c0 + 32 .. c0 + 32 + kKPT - 1 with lanes 16-31 (tcgen05.ld
    // 16x32bx2), lane i and i + 16 holding row 16 sp + i. The warps of a row all
    // keep its reference max; it moves only when a score exceeds it by the
    // threshold. P is computed with the current reference first and recomputed
    // by a warp with a row whose reference moves (rare: the first visible keys,
    // a large new score), once every part's maximum has been exchanged.
    const int si = warp - 2;                        // 0 .. kSoftmaxWarps - 1
    const int sp = warp & 3;                        // TMEM sub-partition
    const int kw = si >> 2;                         // which part of the keys
    constexpr int kParts = kKeyWarps / 2;           // parts per 64-key half
    const int c0 = 64 * (kw / kParts) + kKPT * (kw % kParts);   // first column of lanes 0-15
    const uint32_t lane_base = static_cast<uint32_t>(32 * sp) << 16;
    const int row = 16 * sp + (lane & 15);
    const int kq = lane >> 4;
    const bool live = row < R;
    // last key (sequence-relative) this row may see inside this split: bottom-right causal
    const int lim_r = live ? min(key_end - 1, kvlen - sq + row / group) : -1;
    const float sc = dq * dk * a.scale_log2;
    // With a positive score scale the max is taken on the raw scores and the
    // scale goes into the exponent's FMA (esc = sc); otherwise the scores are
    // scaled as they are loaded (esc = 1).
    const bool raw_ok = sc > 0.f;
    const float esc = raw_ok ? sc : 1.f;
    float* hmax = reinterpret_cast<float*>(smem + kOffHalf);   // [2 tile parity][kKeyWarps][64 rows]
    float* hsum = hmax + 2 * kKeyWarps * 64;                     // [kKeyWarps][64 rows]
    volatile int* wflags = reinterpret_cast<volatile int*>(smem + kOffFlags);   // [2][kSoftmaxWarps], then bad
    float m_run = -INFINITY;   // the row's reference max (log2 units), kept by all of its lanes
    float lsum = 0.f;          // fp32 softmax denominator over this thread's keys
    int bad = 0;
    // this thread's kKPT scores of tile t (S buffer t & 1), times esc in log2
    // units (raw when esc = sc), -inf where not visible; returns their max (in the
    // same units)
    auto load_scores = [&](int t, bool w, float (&x)[kKPT]) -> float {
      uint32_t raw[kKPT];
      const uint32_t col = tmem + lane_base + kTmemS + 128 * (t & 1) + c0;
      tld_16x32bx2_h32(col, raw);
      twait_ld(raw);
      const int key0 = (tile0 + t) * kTile + c0 + 32 * kq;   // sequence-relative
      const float ls = raw_ok ? 1.f : sc;
      float mx = -INFINITY;
      if (w && key0 + kKPT - 1 <= lim_r) {
        if (raw_ok) {
#pragma unroll
          for (int i = 0; i < kKPT; ++i) x[i] = __uint_as_float(raw[i]);
        } else {
#pragma unroll
          for (int i = 0; i < kKPT; ++i) x[i] = __uint_as_float(raw[i]) * sc;
        }
        mx = max32(x);
      } else if (w) {
#pragma unroll
        for (int i = 0; i < kKPT; ++i) {
          x[i] = key0 + i <= lim_r ? __uint_as_float(raw[i]) * ls : -INFINITY;
          mx = fmaxf(mx, x[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < kKPT; ++i) x[i] = -INFINITY;
      }
      return mx;
    };
    // p = 2^(x esc - m_ref) as f16 into P: one FMA and one exponential per score,
    // exactly 0 where not visible (x = -inf; while m_ref is still -inf the
    // reference is taken as 0, and a row with a visible score recomputes P once
    // its reference has moved) (the K-major B operand
    // of PV: N = rows, K = keys; a row's 64 keys of one half are one 128-byte line
    // of that half's swizzle atom, this thread's keys its 16-byte pieces from
    // (c0 % 64 + 32 kq) / 8 on; rows past R are never read back: not stored);
    // returns the sum of p
    const int p_atom = c0 / 64, p_piece = (c0 % 64 + 32 * kq) / 8;
    auto exp_store = [&](int t, const float (&x)[kKPT]) -> float {
      uint32_t h[kKPT / 2];
      float ps[kKPT / 2];
      const float nm = m_run == -INFINITY ? 0.f : -m_run;
#pragma unroll
      for (int i = 0; i < kKPT / 2; ++i) {
        const float p0 = ex2_approx(fmaf(x[2 * i], esc, nm));
        const float p1 = ex2_approx(fmaf(x[2 * i + 1], esc, nm));
        ps[i] = p0 + p1;
        const __half2 ph = __floats2half2_rn(p0, p1);
        h[i] = *reinterpret_cast<const uint32_t*>(&ph);
      }
#pragma unroll
      for (int w2 = kKPT / 4; w2 > 0; w2 >>= 1)
#pragma unroll
        for (int i = 0; i < w2; ++i) ps[i] += ps[i + w2];
      if (live) {
        uint8_t* pt = smem + kOffP + (t % kPBuffers) * kPBytes + p_atom * 8192 + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
        for (int c = 0; c < kKPT / 8; ++c)
          *reinterpret_cast<uint4*>(pt + (((p_piece + c) ^ (row & 7)) << 4)) =
              make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
      }
      return ps[0];
    };
    // the per-tile word of warp kk of sub-partition sub
    auto warp_of = [](int sub, int kk) { return ((sub + 2) & 3) + 4 * kk; };
#pragma unroll 1
    for (int t = 0; t < nt; ++t) {
      int w = 1;
      if (lane == 0) w = wait_bounded(bar(B_SREADY0 + (t & 1)), (t >> 1) & 1, wc, W_SM_S);
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) bad = 1;
      tc_fence_after();
      float x[kKPT];
      float mx = load_scores(t, w != 0, x);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16)) * esc;   // this warp's part of the row, log2 units
      const bool need = mx > m_run + kRescaleThreshold;
      float* alpha = alpha_s + 64 * (t & 1);
      if (lane < 16) {
        hmax[((t & 1) * kKeyWarps + kw) * 64 + row] = mx;
        if (kw == 0) alpha[row] = 1.f;   // rewritten below for a row whose reference moves
      }
      const unsigned rmask = __ballot_sync(0xffffffffu, need) & 0xffffu;
      if (lane == 0) wflags[(t & 1) * kSoftmaxWarps + si] = static_cast<int>(rmask) | (bad ? 0x10000 : 0);
      float ts = exp_store(t, x);   // with the current reference
      // Every warp's maxima and words of this tile are written; the barrier's own
      // reduction says whether any row moves or any wait failed. Only then are
      // the words read (shared-memory loads right after the barrier wait behind
      // the tile's stores).
      const bool report = named_bar_or(1, 32 * kSoftmaxWarps, need || bad != 0);
      uint64_t moving = 0;   // bit r: the reference of row r moves in this tile
      bool failed = false;
      if (report) {
#pragma unroll
        for (int sub = 0; sub < 4; ++sub) {
          int f = 0;
#pragma unroll
          for (int kk = 0; kk < kKeyWarps; ++kk) f |= wflags[(t & 1) * kSoftmaxWarps + warp_of(sub, kk)];
          failed |= (f & 0x10000) != 0;
          moving |= static_cast<uint64_t>(f & 0xffff) << (16 * sub);
        }
      }
      if (failed) {
        bad = 1;
        break;   // every softmax warp sees the same words and leaves together
      }
      const unsigned mv = static_cast<unsigned>(moving >> (16 * sp)) & 0xffffu;   // this warp's rows that move
      if (mv != 0) {
        // a row whose reference moves takes the max of all of its parts; the
        // warp reloads its scores and redoes P and the tile sum (a row that does
        // not move gets the same values again)
        if ((mv >> (lane & 15)) & 1u) {
          float nm = -INFINITY;
#pragma unroll
          for (int kk = 0; kk < kKeyWarps; ++kk) nm = fmaxf(nm, hmax[((t & 1) * kKeyWarps + kk) * 64 + row]);
          const float al = (m_run == -INFINITY) ? 0.f : ex2_approx(m_run - nm);
          lsum *= al;
          m_run = nm;
          if (kw == 0 && lane < 16) alpha[row] = al;
        }
        load_scores(t, w != 0, x);
        ts = exp_store(t, x);
      }
      lsum += ts;
      if (moving != 0 && t >= 1) {
        // O^T holds PV of earlier tiles: once PV(t-1) is done, scale the columns
        // (rows) that moved, in this warp's 32 dims (TMEM lanes) and its kCPW of
        // the 64 columns, after every warp has written its factors
        named_bar_sync(1, 32 * kSoftmaxWarps);
        int wp = 1;
        if (lane == 0) wp = wait_bounded(bar(B_PVDONE), (t - 1) & 1, wc, W_SM_PV);
        if (!__shfl_sync(0xffffffffu, wp, 0)) bad = 1;
        tc_fence_after();
        const unsigned mc = static_cast<unsigned>(moving >> (kCPW * kw)) &
                            static_cast<unsigned>((1ull << kCPW) - 1);
        if (mc != 0 && !bad) {
          uint32_t o[kCPW];
          tld_32x32b(tmem + lane_base + kCPW * kw, o);
          twait_ld(o);
#pragma unroll
          for (int i = 0; i < kCPW; ++i)
            if ((mc >> i) & 1u) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha[kCPW * kw + i]);
          tst_32x32b(tmem + lane_base + kCPW * kw, o);
          tmem_wait_st();
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL0 + (t & 1)));
      // alpha, the maxima and the words of this tile's parity are rewritten two
      // tiles on, before the first named barrier of that tile, which every warp
      // reaches only after it has read them here
    }

    // ---- epilogue ---------------------------------------------------------
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);   // this warp's part of the row
    if (lane == 0) wflags[2 * kSoftmaxWarps + si] = bad;
    if (lane < 16) hsum[kw * 64 + row] = lsum;
    named_bar_sync(1, 32 * kSoftmaxWarps);
    int any_bad = 0;
#pragma unroll
    for (int k = 0; k < kSoftmaxWarps; ++k) any_bad |= wflags[2 * kSoftmaxWarps + k];
    if (kw == 0 && lane < 16 && live) {
      float tot = 0.f;   // every part of the row
#pragma unroll
      for (int kk = 0; kk < kKeyWarps; ++kk) tot += hsum[kk * 64 + row];
      float lse = -INFINITY, inv = 0.f;
      if (tot > 0.f) {
        lse = m_run + log2f(tot);
        inv = dv / tot;
      }
      inv_s[row] = inv;
      if (!any_bad) {
        if (direct) {
          if (a.lse_out != nullptr) a.lse_out[out_index(row)] = lse;
        } else {
          a.lse_acc[out_index(row)] = lse;
        }
      }
    }
    named_bar_sync(1, 32 * kSoftmaxWarps);
    if (!any_bad) {
      int w = 1;
      if (lane == 0) w = wait_bounded(bar(B_FINAL), 0, wc, W_SM_FINAL);
      w = __shfl_sync(0xffffffffu, w, 0);
      tc_fence_after();
      if (w) {
        // O^T: this thread's dim d (a TMEM lane) of the warp's kCPW rows (columns)
        uint32_t o[kCPW];
        tld_32x32b(tmem + lane_base + kCPW * kw, o);
        twait_ld(o);
        const int d = 32 * sp + lane;
        float amax_l = 0.f;
        float inv[kCPW];   // in registers: no shared-memory reload between the global stores
#pragma unroll
        for (int j = 0; j < kCPW; ++j) inv[j] = inv_s[kCPW * kw + j];
#pragma unroll
        for (int j = 0; j < kCPW; ++j) {
          const int rho = kCPW * kw + j;
          if (rho >= R) continue;
          const float v = __uint_as_float(o[j]) * inv[j];
          const size_t oi = out_index(rho) * kD + d;
          if (!direct) {
            a.o_acc[oi] = v;
          } else {
            amax_l = fmaxf(amax_l, fabsf(v));
            if (a.out_dtype == 0) {
              static_cast<float*>(a.out)[oi] = v;
            } else if (a.out_dtype == 1) {
              static_cast<__nv_bfloat16*>(a.out)[oi] = __float2bfloat16_rn(v);
            } else {
              static_cast<uint8_t*>(a.out)[oi] =
                  static_cast<uint8_t>(__nv_cvt_float_to_fp8(v * a.inv_scale, __NV_SATFINITE, __NV_E4M3));
            }
          }
        }
        if (direct && a.amax != nullptr) {
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) amax_l = fmaxf(amax_l, __shfl_xor_sync(0xffffffffu, amax_l, o2));
          if (lane == 0) atomicMax(reinterpret_cast<int*>(a.amax), __float_as_int(amax_l));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int sdpa_decode_smem_bytes() { return kSmemBytes; }

cudaError_t prepare_sdpa_kernels() {
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  return cudaFuncSetAttribute(sdpa_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_sdpa_decode(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                               const SdpaArgs& a, bool direct, cudaStream_t stream) {
  // adaptive: at most num_sms jobs, unless every sequence has one split
  const long long all = static_cast<long long>(a.batch) * a.h_kv * a.num_splits;
  const long long one = static_cast<long long>(a.batch) * a.h_kv;
  const long long bound = a.adaptive ? (one > a.num_sms ? one : static_cast<long long>(a.num_sms)) : all;
  const dim3 grid(static_cast<unsigned>(bound < all ? bound : all));
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, sdpa_decode_kernel, tm_q, tm_k, tm_v, a, direct ? 1 : 0);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace skv

// Split-KV sparse-MLA decode kernel for sm_103a (tcgen05 MMAs, TMEM accumulators,
// cp.async row gathers).
//
// What one CTA computes (FlashMLA PR #25, "What changes"): the job
// (query token t, KV split s) walks the top-k entries [row0, row1) of its own
// block range, gathers those rows of the shared latent KV cache, and produces
// for each of the 64 heads either
//   split path:  O_acc = sum_r e^{s_r} V_r / sum_r e^{s_r} (fp32) and the log2 LSE,
//   direct path: the same O with the attention sink folded into the
//                denominator, cast to fp32 / bf16 / e4m3, plus LSE and amax.
//
// Layout of the work (one CTA per job, 256 threads, 64 gathered rows per step):
//   warps 0-2  loads: Q once by TMA (9 tiles of 64 heads x 64 dims); per step
//              the 64 gathered rows as 4608 16-byte cp.async copies (each row
//              is 72 contiguous 16-byte pieces; a warp instruction covers 512
//              contiguous bytes of a row), written in the 128-byte-swizzled
//              layout into one half of a ring of two 64-row halves; an invalid
//              index copies zeros and reads nothing. Completion is tracked per
//              thread by cp.async.mbarrier.arrive.
//   warp 3     tcgen05 issue (one thread), all descriptors precomputed:
//                S[64 heads x 64 rows]  = Q . K_half^T                  (M=64, N=64, K=576)
//                O^T[512 x 64 heads]   += V_half^T . (P_hi + P_lo)^T    (4 x (M=128, N=64, K=64), twice)
//              V is read straight out of the gathered rows as an MN-major
//              operand; Q, K and P^T are K-major; all tiles use the 128-byte
//              swizzle. Each QK and each PV is one unbroken run of MMAs.
//   warps 4-7  softmax: an M=64 accumulator keeps head 16w+i in lane i of TMEM
//              sub-partition w, so warp 4+w owns heads 16w..16w+15; its lanes
//              0-15 take rows 0-31 and lanes 16-31 rows 32-63 of the step (one
//              16x32bx2 TMEM load). A head's running max and row sum live in two
//              lanes of one warp; only a rescale of O^T (rare, lazy) is shared
//              with the other warps, through a per-step barrier that is arrived
//              on early and waited on late. Then the epilogue.
//
// Precision: p = 2^(x - m_ref) is stored as P_hi = p truncated to bf16 and
// P_lo = bf16(p - P_hi); the PV product uses both, so P enters O with ~2^-15
// relative error instead of the 2^-8 of a single bf16. The fp32 sum of p (the
// softmax denominator, and the LSE) stays in per-thread partials, reduced once
// at the end; it matches the P the product used to the same ~2^-15.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"
#include "softmax_util.cuh"

namespace skv {
namespace {

constexpr int kThreads = 256;
constexpr int kProducers = 96;                      // warps 0-2
constexpr int kPiecesPerRow = 72;                   // 1152 B / 16 B
constexpr int kPiecesPerThread = kMlaBlockRows * kPiecesPerRow / kProducers;   // 48
constexpr int kChunks = 9;                          // 576 dims = 9 column chunks of 64 (128 B)
constexpr int kSlotBytes = 16384;                   // one column chunk of both halves
constexpr int kHalfBytes = 8192;                    // one column chunk of one 64-row half
constexpr int kQChunkBytes = 8192;                  // 64 heads x 128 B
constexpr int kRingBytes = kChunks * kSlotBytes;    // 147456
constexpr int kQBytes = kChunks * kQChunkBytes;     // 73728

// Shared memory map. The dynamic shared memory base is 1024-byte aligned (the
// kernel checks it and refuses to run otherwise), so no slack is reserved.
constexpr int kOffRing = 0;
constexpr int kOffQ = kOffRing + kRingBytes;        // 147456
constexpr int kOffPlo = kOffQ + kQBytes;            // 221184: P_lo, 64 rows x 64 heads bf16
constexpr int kOffBars = kOffPlo + kHalfBytes;      // 229376
constexpr int kOffMisc = kOffBars + 128;            // [0] tmem base, [1] abort flag, [2..3] go,
                                                    // [4..11] rescale masks [2][4], [12..15] final flags
constexpr int kOffAlpha = kOffMisc + 128;           // float[2][64] rescale factors by step parity
constexpr int kOffInv = kOffAlpha + 512;            // float[64] 1/denominator (epilogue)
constexpr int kOffIdx = kOffInv + 1024;             // int[2][64] row indices of the step, per half
constexpr int kSmemBytes = kOffIdx + 512;           // 231680

enum {
  B_QFULL = 0, B_FULL0, B_FULL1, B_EMPTY0, B_EMPTY1, B_SFULL0, B_SFULL1,
  B_PFULL0, B_PFULL1, B_PVDONE, B_DRAIN, B_XCH0, B_XCH1, kNumBars
};
static_assert(kNumBars * 8 <= 128, "barrier area");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 256;                    // S^T buffers at columns 256 and 320
constexpr float kRescaleThreshold = 8.0f;           // p = 2^(x - m_ref) <= 256 between rescales
constexpr float kLog2e = 1.4426950408889634f;

// Wait sites reported in the status word when a bounded wait runs out.
enum : uint32_t {
  W_PROD_EMPTY = 1, W_MMA_Q, W_MMA_STALL, W_SM_S, W_SM_PV, W_SM_PV_EPI, W_DRAIN_MMA, W_SM_X
};

// 128-byte-swizzled byte offset of the 16-byte piece `piece` (0-7) of row `row`
// inside a tile of 128-byte rows grouped in 1024-byte, 8-row atoms.
__device__ __forceinline__ int sw128(int row, int piece) {
  return (row >> 3) * 1024 + (row & 7) * 128 + ((piece ^ (row & 7)) << 4);
}

template <bool kDirect>
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const MlaArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- job decode: one place, shared by every role --------------------------
  const int t = blockIdx.x / a.num_splits;
  const int s = blockIdx.x - t * a.num_splits;
  const int base = a.num_blocks / a.num_splits;
  const int rem = a.num_blocks - base * a.num_splits;
  const int blk0 = s * base + min(s, rem);
  const int nblk = base + (s < rem ? 1 : 0);
  const int row0 = min(blk0 * kMlaBlockRows, a.topk);
  const int row1 = min((blk0 + nblk) * kMlaBlockRows, a.topk);
  const int nsteps = (row1 - row0 + kMlaBlockRows - 1) / kMlaBlockRows;
  const size_t out_row = kDirect ? static_cast<size_t>(t) * kMlaHeads
                                 : (static_cast<size_t>(s) * a.s_q + t) * kMlaHeads;

  if (nsteps == 0) {
    // A split with no block of its own: O = 0, LSE = -inf (only the split path
    // can have one; the direct path always has topk >= 1 entries).
    grid_launch_dependents();
    float4* o = reinterpret_cast<float4*>(a.o_acc + out_row * kMlaDv);
    for (int i = threadIdx.x; i < kMlaHeads * kMlaDv / 4; i += kThreads)
      o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (threadIdx.x < kMlaHeads) a.lse_acc[out_row + threadIdx.x] = -INFINITY;
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
  volatile int* fin = reinterpret_cast<volatile int*>(misc + 12);             // [4] final per-warp flags
  float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
  float* inv_s = reinterpret_cast<float*>(smem + kOffInv);
  const WaitCtx wc{a.wait_limit_ns, a.status, abort_flag};
  const int32_t* idx_t = a.idx + static_cast<size_t>(t) * a.topk;

  // The first row indices: fetched before the set-up barrier so the global
  // memory latency overlaps TMEM allocation and barrier initialisation. Loader
  // thread i < 64 takes row i of step 0; every softmax warp takes rows lane and
  // lane + 32 of step 0.
  int first_idx = -1, first_idx2 = -1;
  {
    int r = -1;
    if (threadIdx.x < kMlaBlockRows) r = row0 + static_cast<int>(threadIdx.x);
    if (warp >= 4) r = row0 + lane;
    if (r >= 0 && r < row1) first_idx = __ldg(idx_t + r);
    if (warp >= 4 && r + 32 < row1) first_idx2 = __ldg(idx_t + r + 32);
    if (first_idx < 0 || first_idx >= a.n_kv) first_idx = -1;
  }

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_FULL0), kProducers);   // one cp.async completion arrival per producer thread
    mbar_init(bar(B_FULL1), kProducers);
    mbar_init(bar(B_EMPTY0), 1);
    mbar_init(bar(B_EMPTY1), 1);
    mbar_init(bar(B_SFULL0), 1);
    mbar_init(bar(B_SFULL1), 1);
    mbar_init(bar(B_PFULL0), 4);
    mbar_init(bar(B_PFULL1), 4);
    mbar_init(bar(B_PVDONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_XCH0), 4);             // one arrival per softmax warp
    mbar_init(bar(B_XCH1), 4);
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
  // The combine (a programmatic dependent) may begin launching now; it waits
  // for this whole grid to finish before it reads any partial.
  grid_launch_dependents();

  if (warp < 3) {
    // ========================================================== loaders ===
    const int ptid = threadIdx.x;          // 0..95
    int* idx_s = reinterpret_cast<int*>(smem + kOffIdx);
    volatile int* go = reinterpret_cast<volatile int*>(misc + 2);   // [2]: by step parity
    if (ptid == 0) {
      tma_prefetch_desc(&tm_q);
      mbar_arrive_expect_tx(bar(B_QFULL), kQBytes);
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c)
        tma_load_2d(sbase + kOffQ + c * kQChunkBytes, &tm_q, 64 * c, kMlaHeads * t, bar(B_QFULL));
    }
    // thread ptid < 64 fetches the row index of row ptid of a step
    auto fetch = [&](int k) -> int {
      const int r = row0 + kMlaBlockRows * k + ptid;
      int v = -1;
      if (ptid < kMlaBlockRows && r < row1) {
        v = __ldg(idx_t + r);
        if (v < 0 || v >= a.n_kv) v = -1;
      }
      return v;
    };
    int cur = first_idx;
#pragma unroll 1
    for (int k = 0; k < nsteps; ++k) {
      const int h = k & 1;
      const int nxt = (k + 1 < nsteps) ? fetch(k + 1) : -1;   // in flight during the wait below
      if (ptid < kMlaBlockRows) idx_s[h * kMlaBlockRows + ptid] = cur;
      if (ptid == 0) go[h] = (k < 2) ? 1 : wait_bounded(bar(B_EMPTY0 + h), ((k >> 1) - 1) & 1, wc, W_PROD_EMPTY);
      named_bar_sync(2, kProducers);     // the half is free and its row indices are visible
      if (!go[h]) break;                 // every loader sees the same flag
      const uint32_t half_base = sbase + kOffRing + h * kHalfBytes;
      // all index reads first: a read after a cp.async (which writes shared
      // memory) would have to wait for it
      int ixr[kPiecesPerThread];
#pragma unroll
      for (int i = 0; i < kPiecesPerThread; ++i) ixr[i] = idx_s[h * kMlaBlockRows + (ptid + kProducers * i) / kPiecesPerRow];
#pragma unroll
      for (int i = 0; i < kPiecesPerThread; ++i) {
        const int u = ptid + kProducers * i;
        const int row = u / kPiecesPerRow;
        const int seg = u - row * kPiecesPerRow;
        const int ix = ixr[i];
        const uint32_t dst = half_base + (seg >> 3) * kSlotBytes + sw128(row, seg & 7);
        const uint8_t* src = a.kv + static_cast<size_t>(ix < 0 ? 0 : ix) * (kMlaDqk * 2) + seg * 16;
        cp_async_16(dst, src, ix < 0 ? 0u : 16u);
      }
      cp_async_arrive_noinc(bar(B_FULL0 + h));
      cur = nxt;
    }
    cp_async_wait_all();   // nothing of this thread is still landing when the CTA exits
  } else if (warp == 3) {
    // ========================================================= MMA issuer ===
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_make(64, 64, 1, false, false);   // A (Q), B (K rows) K-major
      constexpr uint32_t kIdescPV = idesc_make(128, 64, 1, true, false);   // A (V^T) MN-major, B (P^T) K-major
      // Descriptors of the operands' first K step; every other one differs only
      // in the start-address field (bits 0-13, address >> 4, no carry out of it
      // below 256 KB), so the issue loop adds a constant.
      // (half 1 is half 0 shifted by kHalfBytes)
      const uint64_t d_k0 = sdesc_sw128(sbase + kOffRing, 16, 1024);
      const uint64_t d_v0 = sdesc_sw128(sbase + kOffRing, kSlotBytes, 1024);
      const uint64_t d_phi0 = sdesc_sw128(sbase + kOffRing + 8 * kSlotBytes, 16, 1024);
      constexpr uint64_t kHalfStep = kHalfBytes >> 4;
      const uint64_t d_q = sdesc_sw128(sbase + kOffQ, 16, 1024);
      const uint64_t d_plo = sdesc_sw128(sbase + kOffPlo, 16, 1024);
      // QK(k): 9 column chunks of 64 dims x 4 MMAs of K=16 (32 bytes of a K-major
      // row each), issued back to back with constant descriptor offsets
      auto issue_qk = [&](int k) {
        const uint32_t d = tmem + kTmemS + 64 * (k & 1);
        const uint64_t ak = d_k0 + (k & 1) * kHalfStep;
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16(d, d_q + (c * kQChunkBytes) / 16 + 2 * kk, ak + (c * kSlotBytes) / 16 + 2 * kk, kIdescQK,
                    (c | kk) != 0);
      };
      // PV(k): for each 128-dim tile j of V, K = the 64 rows in 4 steps of 16
      // (2048 B of the MN-major V^T, 32 B of the K-major P^T each), first with
      // P_hi, then with P_lo.
      auto issue_pv = [&](int k) {
        const uint64_t av = d_v0 + (k & 1) * kHalfStep;
        const uint64_t bphi = d_phi0 + (k & 1) * kHalfStep;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint64_t bp = part ? d_plo : bphi;
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16(tmem + 64 * j, av + (2 * j * kSlotBytes + kk * 2048) / 16, bp + 2 * kk, kIdescPV,
                      (k > 0 || part > 0 || kk > 0));
        }
      };
      bool ok = wait_bounded(bar(B_QFULL), 0, wc, W_MMA_Q);
      // PV(k) is issued as soon as softmax(k) has written P: its completion
      // frees the half for the loads of step k+2, the loop's critical chain.
      // QK(k) is issued once its rows have landed and its S^T buffer is free
      // (softmax(k-2) is done, i.e. PV(k-2) was issued). tcgen05 runs them in
      // issue order, each as one unbroken run of MMAs: instructions between two
      // MMAs of a run stall the tensor pipe. When only one of the two can make
      // progress the thread sleeps in try_wait on that barrier; otherwise it
      // polls both.
      int nqk = 0, npv = 0;
      uint64_t t_idle = 0;
      while (ok && npv < nsteps) {
        const bool can_pv = npv < nqk;
        const bool can_qk = nqk < nsteps && nqk <= npv + 1;
        const uint32_t pbar = bar(B_PFULL0 + (npv & 1)), pph = (npv >> 1) & 1;
        const uint32_t fbar = bar(B_FULL0 + (nqk & 1)), fph = (nqk >> 1) & 1;
        bool progress = false;
        if (can_pv && (can_qk ? mbar_test_wait(pbar, pph) : mbar_try_wait(pbar, pph))) {
          tc_fence_after();
          issue_pv(npv);
          mma_commit(bar(B_EMPTY0 + (npv & 1)));
          mma_commit(bar(B_PVDONE));
          ++npv;
          progress = true;
        } else if (can_qk && (can_pv ? mbar_test_wait(fbar, fph) : mbar_try_wait(fbar, fph))) {
          // the rows were written by other threads' cp.async (generic proxy);
          // make them visible to the tensor core's reads (async proxy)
          fence_proxy_async_smem();
          tc_fence_after();
          issue_qk(nqk);
          mma_commit(bar(B_SFULL0 + (nqk & 1)));
          ++nqk;
          progress = true;
        }
        if (progress) {
          t_idle = 0;
        } else {
          const uint64_t now = globaltimer_ns();
          if (*abort_flag) {
            ok = false;
          } else if (t_idle == 0) {
            t_idle = now;
          } else if (now - t_idle > a.wait_limit_ns) {
            *abort_flag = 1;
            atomicOr(&a.status[0], 1u);
            atomicCAS(&a.status[1], 0u, W_MMA_STALL);
            ok = false;
          }
        }
      }
      if (!ok) {
        // no MMA may still be reading shared memory or writing TMEM when the CTA exits
        mma_commit(bar(B_DRAIN));
        if (!wait_drain(bar(B_DRAIN), 0, a.wait_limit_ns)) atomicCAS(&a.status[1], 0u, W_DRAIN_MMA);
      }
    }
  } else {
    // ============================================== softmax + epilogue ====
    const int sp = warp & 3;               // TMEM sub-partition (lanes 32sp..32sp+31)
    const int tid = threadIdx.x - 128;     // 0..127
    const uint32_t lane_base = static_cast<uint32_t>(32 * sp) << 16;
    const int head = 16 * sp + (lane & 15);   // this thread's head
    const int rb = (lane >> 4) * 32;          // and its 32 rows rb..rb+31 of every step
    float m_run = -INFINITY;   // reference max of the head (log2 units), shared by its two lanes
    float lsum = 0.f;          // fp32 softmax denominator over this thread's rows
    int bad = 0;               // a bounded wait of this warp ran out
    int ia = first_idx, ib = first_idx2;   // indices of rows lane and lane + 32 of the step

#pragma unroll 1
    for (int k = 0; k < nsteps; ++k) {
      const int h = k & 1;
      // which of this thread's 32 rows hold a valid index
      const uint32_t vlo = __ballot_sync(0xffffffffu, ia >= 0 && ia < a.n_kv);
      const uint32_t vhi = __ballot_sync(0xffffffffu, ib >= 0 && ib < a.n_kv);
      const uint32_t vm = rb ? vhi : vlo;
      if (k + 1 < nsteps) {   // the next step's indices, in flight during this step
        const int rn = row0 + kMlaBlockRows * (k + 1) + lane;
        ia = rn < row1 ? __ldg(idx_t + rn) : -1;
        ib = rn + 32 < row1 ? __ldg(idx_t + rn + 32) : -1;
      }

      int w = 1;
      if (lane == 0) w = wait_bounded(bar(B_SFULL0 + h), (k >> 1) & 1, wc, W_SM_S);
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) bad = 1;
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
        float t[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) t[i] = x[i] + x[i + 16];
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] += t[i + 8];
#pragma unroll
        for (int i = 0; i < 4; ++i) t[i] += t[i + 4];
        lsum += (t[0] + t[2]) + (t[1] + t[3]);
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
      int wx = 1;
      if (lane == 0) wx = wait_bounded(bar(B_XCH0 + h), (k >> 1) & 1, wc, W_SM_X);
      wx = __shfl_sync(0xffffffffu, wx, 0);
      if (!wx) bad = 1;
      const uint32_t x0 = xch[h * 4 + 0], x1 = xch[h * 4 + 1], x2 = xch[h * 4 + 2], x3 = xch[h * 4 + 3];
      if (((x0 | x1 | x2 | x3) & 0x10000u) || !wx) {
        bad = 1;
        break;   // every softmax warp sees the same masks and leaves together
      }
      // PV(k-1) must be complete before O^T is rescaled and before P_lo (one
      // buffer for all steps) is overwritten.
      if (k >= 1) {
        int wp = 1;
        if (lane == 0) wp = wait_bounded(bar(B_PVDONE), (k - 1) & 1, wc, W_SM_PV);
        wp = __shfl_sync(0xffffffffu, wp, 0);
        if (!wp) bad = 1;
        tc_fence_after();
        const uint64_t resc = static_cast<uint64_t>(x0) | (static_cast<uint64_t>(x1) << 16) |
                              (static_cast<uint64_t>(x2) << 32) | (static_cast<uint64_t>(x3) << 48);
        if (resc != 0 && !bad) {
          // O^T holds PV of steps < k: scale the columns of the rescaled heads
          // in the 32 dims (TMEM lanes) of each tile this warp can reach
#pragma unroll 1
          for (int j = 0; j < 8; ++j) {   // 4 O^T tiles x 2 halves of 32 head columns
            const int c0 = 32 * (j & 1);
            if (((resc >> c0) & 0xffffffffull) == 0) continue;
            uint32_t o[32];
            float al[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) al[i] = ((resc >> (c0 + i)) & 1ull) ? alpha_s[h * 64 + c0 + i] : 1.f;
            const uint32_t col = 64 * (j >> 1) + c0;
            tmem_ld_32x32b_x32(tmem + lane_base + col, o);
            tmem_wait_ld_x32(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * al[i]);
            tmem_st_32x32b_x32(tmem + lane_base + col, o);
          }
          tmem_wait_st();
        }
      }
      // P^T as a K-major operand: N = heads, K = rows; the 64 rows of one head
      // are one 128-byte line of the swizzled tile, this thread's 32 rows are
      // its pieces rb/8 .. rb/8+3.
      {
        uint8_t* p_hi = smem + kOffRing + 8 * kSlotBytes + h * kHalfBytes;
        uint8_t* p_lo = smem + kOffPlo;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int off = sw128(head, (rb >> 3) + q);
          *reinterpret_cast<uint4*>(p_hi + off) = make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
          *reinterpret_cast<uint4*>(p_lo + off) = make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL0 + h));
    }

    // ---- epilogue ---------------------------------------------------------
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
    if (lane == 0) fin[sp] = bad;
    if (lane < 16) {
      float lse = -INFINITY, inv = 0.f;
      if (lsum > 0.f) {
        lse = m_run + log2f(lsum);
        float den = lsum;
        if (kDirect && a.sink != nullptr) den += exp2f(a.sink[head] * kLog2e - m_run);
        inv = 1.f / den;
      }
      inv_s[head] = inv;
      if (kDirect) {
        if (a.lse_out != nullptr) a.lse_out[out_row + head] = lse;
      } else {
        a.lse_acc[out_row + head] = lse;
      }
    }
    named_bar_sync(1, 128);
    const bool any_bad = fin[0] | fin[1] | fin[2] | fin[3];
    int wp = 0;
    if (!any_bad) {
      if (lane == 0) wp = wait_bounded(bar(B_PVDONE), (nsteps - 1) & 1, wc, W_SM_PV_EPI);
      wp = __shfl_sync(0xffffffffu, wp, 0);
      tc_fence_after();
    }
    if (!any_bad && wp) {
      // Stage the [64 heads][512] output tile in the ring (free now: every load
      // has landed and every MMA has completed), then copy it to global memory
      // with one bulk copy; a job's output rows are contiguous there.
      float amax_l = 0.f;
      float inv[64];   // in registers: no shared-memory reload between the stores
#pragma unroll
      for (int c = 0; c < 64; ++c) inv[c] = inv_s[c];
      const int esize = (!kDirect || a.out_dtype == 0) ? 4 : (a.out_dtype == 1 ? 2 : 1);
      uint8_t* stage = smem + kOffRing;
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        uint32_t o[64];
        tmem_ld_32x32b_x64(tmem + lane_base + 64 * j, o);
        tmem_wait_ld_x64(o);
        const int d = 128 * j + 32 * sp + lane;
        if (esize == 4) {
          float* st = reinterpret_cast<float*>(stage) + d;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float v = __uint_as_float(o[c]) * inv[c];
            amax_l = fmaxf(amax_l, fabsf(v));
            st[c * kMlaDv] = v;
          }
        } else if (esize == 2) {
          __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(stage) + d;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float v = __uint_as_float(o[c]) * inv[c];
            amax_l = fmaxf(amax_l, fabsf(v));
            st[c * kMlaDv] = __float2bfloat16_rn(v);
          }
        } else {
          uint8_t* st = stage + d;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float v = __uint_as_float(o[c]) * inv[c];
            amax_l = fmaxf(amax_l, fabsf(v));
            st[c * kMlaDv] =
                static_cast<uint8_t>(__nv_cvt_float_to_fp8(v * a.inv_scale, __NV_SATFINITE, __NV_E4M3));
          }
        }
      }
      fence_proxy_async_smem();          // the bulk copy reads the tile through the async proxy
      named_bar_sync(1, 128);
      if (tid == 0) {
        uint8_t* gdst = kDirect ? static_cast<uint8_t*>(a.out) + out_row * kMlaDv * esize
                                : reinterpret_cast<uint8_t*>(a.o_acc + out_row * kMlaDv);
        bulk_store(gdst, sbase + kOffRing, kMlaHeads * kMlaDv * esize);
        bulk_commit_and_wait_all();
      }
      if (kDirect && a.amax != nullptr) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax_l = fmaxf(amax_l, __shfl_xor_sync(0xffffffffu, amax_l, o));
        if (lane == 0) atomicMax(reinterpret_cast<int*>(a.amax), __float_as_int(amax_l));
      }
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
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mla_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_mla_decode(const CUtensorMap& tm_q, const MlaArgs& a, bool direct, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(a.s_q) * static_cast<unsigned>(a.num_splits));
  if (direct)
    mla_decode_kernel<true><<<grid, kThreads, kSmemBytes, stream>>>(tm_q, a);
  else
    mla_decode_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(tm_q, a);
  return cudaGetLastError();
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

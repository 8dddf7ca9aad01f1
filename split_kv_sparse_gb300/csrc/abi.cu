// extern "C" entry points of include/mla_split.h: planning, argument checks,
// TMA descriptor encoding and kernel launches. No entry point allocates device
// memory; the only device state is the per-device status word below.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <atomic>
#include <mutex>

#include "kernels.h"
#include "mla_split.h"

namespace {

using skv::kMlaBlockRows;
using skv::kMlaDqk;
using skv::kMlaDv;
using skv::kMlaHeads;

// [0] = MLA_STATUS_* bits, [1] = code of the first wait that ran out.
__device__ uint32_t g_status[2];

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far above any legitimate wait
// The limit the decode kernels give their pipeline waits (mla_set_wait_limit_ns
// shortens it for tests); an aborting CTA always waits up to kWaitLimitNs for its
// own copies and MMAs in flight.
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};
// 1: the sparse-MLA kernels report indices outside {-1} and [0, n_kv)
// (mla_set_index_checks); 0 by default.
std::atomic<int> g_check_idx{0};
constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  uint32_t* status = nullptr;
  int num_sms = 0;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;

int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MLA_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& d = g_devices[dev];
  if (!d.ready) {
    int major = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_NO_DEVICE;
    }
    if (major != 10) return MLA_ERR_NO_DEVICE;   // the kernels are built for the sm_100 family (sm_103a)
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    if (skv::prepare_mla_kernels() != cudaSuccess || skv::prepare_sdpa_kernels() != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    d.status = static_cast<uint32_t*>(p);
    d.ready = true;
  }
  *out = &d;
  return MLA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_encode_tried) {
    g_encode_tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    } else {
      cudaGetLastError();
    }
  }
  return g_encode;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// Workspace of the (token, split) schedule: fp32 O partials [S][s_q][64][512],
// then fp32 LSE partials [S][s_q][64] at the next 256-byte boundary.
uint64_t split_workspace_bytes(int S, int s_q, int o_elem_bytes = 4) {
  const uint64_t o = static_cast<uint64_t>(S) * s_q * kMlaHeads * kMlaDv * static_cast<uint64_t>(o_elem_bytes);
  return round_up(round_up(o, 256) + static_cast<uint64_t>(S) * s_q * kMlaHeads * 4ull, 256);
}

// Blocks per CTA of the balanced schedule for s_q tokens (0 when it does not
// apply: fewer than 2 blocks per CTA, i.e. every block its own piece).
int64_t balanced_per(int64_t s_q, int nb, int num_sms) {
  const int64_t U = s_q * nb;
  const int64_t per = (U + num_sms - 1) / num_sms;
  return per < 2 ? 0 : per;
}
// CTA ranges of the balanced schedule for s_q tokens: the fewest that reach the
// smallest per-CTA block count on num_sms SMs.
int balanced_ctas(int64_t s_q, int nb, int num_sms) {
  const int64_t U = s_q * nb;
  const int64_t per = (U + num_sms - 1) / num_sms;
  return static_cast<int>((U + per - 1) / per);
}
// The most pieces one token is cut into by the balanced schedule, over every
// s_q up to s_q_max at which the schedule applies: the partial slots its
// workspace needs. Once a CTA range is longer than a token, no token spans more
// than two ranges.
int balanced_slots(int s_q_max, int nb, int num_sms) {
  int most = 1;
  for (int64_t s_q = 1; s_q <= s_q_max; ++s_q) {
    const int64_t per = balanced_per(s_q, nb, num_sms);
    if (per == 0) continue;
    if (per > nb) return std::max(most, 2);
    const int U = static_cast<int>(s_q * nb), P = balanced_ctas(s_q, nb, num_sms);
    for (int64_t t = 0; t < s_q; ++t) {
      const int n = skv::bal_cta_of(static_cast<int>((t + 1) * nb - 1), U, P) -
                    skv::bal_cta_of(static_cast<int>(t * nb), U, P) + 1;
      most = std::max(most, n);
    }
  }
  return most;
}
// The most splits the dense planner's per-sequence rule gives one sequence.
constexpr int kDenseMaxAdaptiveSplits = 16;
// CTAs per (token, split) job: the largest of 4, 2, 1 that still fits `jobs`
// jobs on num_sms SMs at one CTA each.
int dim_groups_for(int64_t jobs, int num_sms) {
  for (int d = 4; d > 1; d /= 2)
    if (jobs * d <= num_sms) return d;
  return 1;
}

// The tail of a one-split grid for s_q tokens, whose last wave would hold r
// tokens: with min(num_blocks, num_sms / r) >= 3 splits those tokens are cut into
// that many splits (*splits; two splits measured no faster than the uncut
// wave); else, when 2 r <= num_sms, each runs whole on two CTAs with half of the
// dims each (*dgroups = 2; full QK, half the PV, final rows, no combine).
// Returns false when the plan or the call has no tail.
bool tail_of(const mla_plan_t* p, int s_q, int* first, int* splits, int* dgroups) {
  if (p->tail_ctas <= 0 || p->num_splits != 1 || s_q <= p->num_sms) return false;
  const int W = p->num_sms, C = std::min(p->tail_ctas, W);
  const int waves = (s_q + W - 1) / W;
  const int r = s_q - (waves - 1) * W;
  const int st = std::min(p->num_blocks, C / r);
  *first = s_q - r;
  *splits = 0;
  *dgroups = 0;
  if (st >= 3) *splits = st;
  else if (2 * r <= C) *dgroups = 2;
  else return false;
  return true;
}

// The workspace of a plan from its split count, schedule and partial type: the
// split layout ([S][s_q_max][64][512] O partials of 4 or 2 bytes, then
// [S][s_q_max][64] fp32 LSE partials at the next 256-byte boundary), large
// enough for the balanced schedule's slots when that schedule is enabled.
void plan_workspace(mla_plan_t* p) {
  const int esz = p->partial_bf16 ? 2 : 4;
  p->o_acc_bytes = p->lse_acc_offset = p->lse_acc_bytes = p->workspace_bytes = 0;
  if (p->num_splits > 1) {
    p->o_acc_bytes = static_cast<uint64_t>(p->num_splits) * p->s_q_max * p->h_q * p->d_v * static_cast<uint64_t>(esz);
    p->lse_acc_offset = round_up(p->o_acc_bytes, 256);
    p->lse_acc_bytes = static_cast<uint64_t>(p->num_splits) * p->s_q_max * p->h_q * 4ull;
    p->workspace_bytes = round_up(p->lse_acc_offset + p->lse_acc_bytes, 256);
  }
  if (p->tail_ctas > 0)   // at most tail_ctas (split, tail token) slots
    p->workspace_bytes = std::max<uint64_t>(p->workspace_bytes, split_workspace_bytes(p->tail_ctas, 1, esz));
  if (p->balanced_ctas > 0)
    p->workspace_bytes = std::max<uint64_t>(
        p->workspace_bytes, split_workspace_bytes(balanced_slots(p->s_q_max, p->num_blocks, p->num_sms), p->s_q_max, esz));
}

int encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  auto enc = encoder();
  if (enc == nullptr) return MLA_ERR_CUDA;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

int encode_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const uint64_t dims_in[3],
              const uint64_t strides_in[2], const uint32_t box_in[3]) {
  auto enc = encoder();
  if (enc == nullptr) return MLA_ERR_CUDA;
  cuuint64_t dims[3] = {dims_in[0], dims_in[1], dims_in[2]};
  cuuint64_t strides[2] = {strides_in[0], strides_in[1]};
  cuuint32_t box[3] = {box_in[0], box_in[1], box_in[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MLA_OK;
  cudaGetLastError();
  return MLA_ERR_CUDA;
}

bool valid_out_dtype(int t) { return t == MLA_OUT_F32 || t == MLA_OUT_BF16 || t == MLA_OUT_E4M3; }

// Shared argument checks of the MLA decode calls.
int check_mla_inputs(int s_q, int topk, const void* q, const void* kv, int64_t n_kv, const int32_t* idx,
                     float sm_scale) {
  if (s_q < 1 || topk < 1) return MLA_ERR_INVALID_ARG;
  if (q == nullptr || kv == nullptr || idx == nullptr) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(idx, 4)) return MLA_ERR_INVALID_ARG;
  if (n_kv < 1 || n_kv > 0x7FFFFFFFll) return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(s_q) * kMlaHeads > 0x7FFFFFFFll) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

int mla_q_tensor_map(int s_q, const void* q, CUtensorMap* tq) {
  return encode_2d(tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, kMlaDqk, static_cast<uint64_t>(s_q) * kMlaHeads,
                   kMlaDqk * 2, 64, 64);
}

}  // namespace

extern "C" {

int mla_abi_version(void) { return MLA_ABI_VERSION; }

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported shape";
    case MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case MLA_ERR_CUDA: return "CUDA call failed";
    case MLA_ERR_NO_DEVICE: return "no usable sm_100-family device";
    default: return "unknown status";
  }
}

int mla_decode_plan(int s_q_max, int h_q, int d_qk, int d_v, int topk, int num_sms, int max_splits,
                    int force_splits, mla_plan_t* out) {
  if (out == nullptr) return MLA_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  if (h_q != kMlaHeads || d_qk != kMlaDqk || d_v != kMlaDv) return MLA_ERR_UNSUPPORTED;
  if (s_q_max < 1 || topk < 1 || num_sms < 0) return MLA_ERR_INVALID_ARG;
  if (max_splits < 0 || max_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
  if (force_splits < MLA_FORCE_BALANCED || force_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
  const bool want_balanced = force_splits == MLA_FORCE_BALANCED;
  if (want_balanced) force_splits = 0;
  if (num_sms == 0) {
    DeviceState* d = nullptr;
    const int st = device_state(&d);
    if (st != MLA_OK) return st;
    num_sms = d->num_sms;
  }
  const int nblk = (topk + kMlaBlockRows - 1) / kMlaBlockRows;
  int S = force_splits;
  if (S == 0) {
    const int cap = max_splits > 0 ? max_splits : MLA_MAX_SPLITS;
    int smax = num_sms / s_q_max;
    if (smax > cap) smax = cap;
    if (smax > nblk) smax = nblk;
    if (smax < 1) smax = 1;
    // A split of two 64-row blocks costs about what a split of one does (the
    // second block's rows land while the first is computed), while every extra
    // split adds a partial to write and to combine and takes SMs the job's dim
    // groups could use: the blocks a split walks count as at least two.
    auto eff_blocks = [&](int c) { return std::max(2, (nblk + c - 1) / c); };
    const int best = eff_blocks(smax);
    S = smax;
    for (int c = 1; c <= smax; ++c)
      if (eff_blocks(c) == best) {
        S = c;
        break;
      }
    // Except when every one-block split still gets 4 dim groups: then a split of
    // one block is quicker than one of two (measured on GB300, topk 640, s_q = 1,
    // 2, 3: 9.2, 9.4, 9.8 us with 10 splits against 10.1, 10.2, 10.5 with 5).
    if (S > 1 && nblk <= smax && static_cast<int64_t>(s_q_max) * nblk * 4 <= num_sms) S = nblk;
  }
  if (static_cast<int64_t>(s_q_max) * S > 0x7FFFFFFFll) return MLA_ERR_INVALID_ARG;
  out->s_q_max = s_q_max;
  out->h_q = h_q;
  out->d_qk = d_qk;
  out->d_v = d_v;
  out->topk = topk;
  out->block_rows = kMlaBlockRows;
  out->num_blocks = nblk;
  out->num_splits = S;
  out->num_sms = num_sms;
  out->dim_groups = dim_groups_for(static_cast<int64_t>(s_q_max) * S, num_sms);
  const int64_t per = balanced_per(s_q_max, nblk, num_sms);
  // The balanced schedule only on request: measured on GB300 (topk 640, back-to-back
  // calls), the uniform grid beat it at every s_q from 96 to 384, even where the
  // grid leaves a wave half empty (s_q = 200: 61.8 us against 87.9 us), since the
  // fp32 partials of the cut tokens, their combine and each CTA's job boundaries
  // cost more than the blocks it saves.
  if (want_balanced && per > 0) {
    // the one-shot call spreads all tokens' blocks over at most num_sms CTAs; its
    // workspace holds a partial slot per piece of the most cut token
    const int64_t units = static_cast<int64_t>(s_q_max) * nblk;
    out->balanced_ctas = static_cast<int32_t>(std::min<int64_t>(units, num_sms));
  }
  // an automatic one-split grid of more than one wave may cut its last wave's tokens
  if (force_splits == 0 && S == 1 && s_q_max > num_sms && nblk >= 2) out->tail_ctas = num_sms;
  plan_workspace(out);
  return MLA_OK;
}

int mla_plan_set_partials_bf16(mla_plan_t* plan, int enable) {
  if (plan == nullptr || (enable != 0 && enable != 1)) return MLA_ERR_INVALID_ARG;
  if (plan->h_q != kMlaHeads || plan->d_v != kMlaDv || plan->num_blocks < 1) return MLA_ERR_INVALID_ARG;
  plan->partial_bf16 = enable;
  plan_workspace(plan);
  return MLA_OK;
}

int mla_sparse_decode_split(const mla_plan_t* plan, int s_q, const void* q, const void* kv, int64_t n_kv,
                            const int32_t* idx, float sm_scale, void* workspace, void* stream) {
  if (plan == nullptr || plan->num_splits < 2 || plan->num_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
  if (plan->h_q != kMlaHeads || plan->d_qk != kMlaDqk || plan->d_v != kMlaDv) return MLA_ERR_UNSUPPORTED;
  if (s_q > plan->s_q_max) return MLA_ERR_INVALID_ARG;
  int st = check_mla_inputs(s_q, plan->topk, q, kv, n_kv, idx, sm_scale);
  if (st != MLA_OK) return st;
  if (workspace == nullptr || !aligned(workspace, 256) || plan->workspace_bytes == 0) return MLA_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != MLA_OK) return st;
  CUtensorMap tq;
  if ((st = mla_q_tensor_map(s_q, q, &tq)) != MLA_OK) return st;
  skv::MlaArgs a{};
  a.kv = static_cast<const uint8_t*>(kv);
  a.idx = idx;
  a.s_q = s_q;
  a.topk = plan->topk;
  a.n_kv = static_cast<int>(n_kv);
  a.num_splits = plan->num_splits;
  a.num_blocks = plan->num_blocks;
  a.dim_groups = plan->dim_groups;
  a.sched = 0;
  a.direct_whole = 0;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.o_acc = static_cast<float*>(workspace);
  a.lse_acc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan->lse_acc_offset);
  a.partial_bf16 = plan->partial_bf16;
  a.status = dev->status;
  a.check_idx = g_check_idx.load();
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.drain_limit_ns = kWaitLimitNs;
  return cuda_status(skv::launch_mla_decode(tq, a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {
// The combine launch shared by the public call (which clears amax itself) and
// the one-shot call (which clears amax before the split pass, so the combine can
// follow the split kernel as a programmatic dependent launch).
int mla_combine_impl(const mla_plan_t* plan, int s_q, const void* workspace, const float* sink, int out_dtype,
                     float out_inv_scale, void* out, float* lse_out, float* amax_out, bool zero_amax,
                     void* stream) {
  if (plan == nullptr || plan->num_splits < 2 || plan->num_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
  if (plan->h_q != kMlaHeads || plan->d_v != kMlaDv) return MLA_ERR_UNSUPPORTED;
  if (s_q < 1 || s_q > plan->s_q_max || out == nullptr || !aligned(out, 16)) return MLA_ERR_INVALID_ARG;
  if (!valid_out_dtype(out_dtype)) return MLA_ERR_INVALID_ARG;
  if (out_dtype == MLA_OUT_E4M3 && !std::isfinite(out_inv_scale)) return MLA_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256) || plan->workspace_bytes == 0) return MLA_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  const int st = device_state(&dev);
  if (st != MLA_OK) return st;
  skv::CombineArgs c{};
  c.o_acc = static_cast<const float*>(workspace);
  c.lse_acc = reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) + plan->lse_acc_offset);
  c.num_splits = plan->num_splits;
  c.partial_bf16 = plan->partial_bf16;
  c.rows = s_q * kMlaHeads;
  c.heads = kMlaHeads;
  c.d = kMlaDv;
  c.sink = sink;
  c.out = out;
  c.out_dtype = out_dtype;
  c.inv_scale = out_inv_scale;
  c.lse_out = lse_out;
  c.amax = amax_out;
  c.num_sms = dev->num_sms;
  return cuda_status(skv::launch_combine(c, zero_amax, /*pdl=*/true, static_cast<cudaStream_t>(stream)));
}

// The one-split grid with its tail cut (tail_of): whole tokens 0 .. tail_first-1
// write their final rows in the decode kernel; the tail tokens' splits write
// partials ([tail_splits][r][64][512], LSE [tail_splits][r][64]) that the
// combine, launched as its programmatic dependent, folds into their rows.
int mla_decode_tail(const mla_plan_t* plan, int s_q, const void* q, const void* kv, int64_t n_kv, const int32_t* idx,
                    float sm_scale, const float* sink, int out_dtype, float out_inv_scale, void* out, float* lse_out,
                    float* amax_out, void* workspace, int tail_first, int tail_splits, void* stream) {
  int st = check_mla_inputs(s_q, plan->topk, q, kv, n_kv, idx, sm_scale);
  if (st != MLA_OK) return st;
  if (out == nullptr || !aligned(out, 16) || !valid_out_dtype(out_dtype)) return MLA_ERR_INVALID_ARG;
  if (out_dtype == MLA_OUT_E4M3 && !std::isfinite(out_inv_scale)) return MLA_ERR_INVALID_ARG;
  const int esz = plan->partial_bf16 ? 2 : 4;
  const int r = s_q - tail_first;
  const uint64_t o_bytes = static_cast<uint64_t>(tail_splits) * r * kMlaHeads * kMlaDv * static_cast<uint64_t>(esz);
  if (workspace == nullptr || !aligned(workspace, 256) ||
      plan->workspace_bytes < split_workspace_bytes(tail_splits, r, esz))
    return MLA_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != MLA_OK) return st;
  CUtensorMap tq;
  if ((st = mla_q_tensor_map(s_q, q, &tq)) != MLA_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (amax_out != nullptr) {
    if ((st = cuda_status(cudaMemsetAsync(amax_out, 0, sizeof(float), cs))) != MLA_OK) return st;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  skv::MlaArgs a{};
  a.kv = static_cast<const uint8_t*>(kv);
  a.idx = idx;
  a.s_q = s_q;
  a.topk = plan->topk;
  a.n_kv = static_cast<int>(n_kv);
  a.num_splits = 1;
  a.num_blocks = plan->num_blocks;
  a.dim_groups = 1;
  a.sched = 0;
  a.direct_whole = 1;
  a.tail_first = tail_first;
  a.tail_splits = tail_splits;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.o_acc = reinterpret_cast<float*>(ws);
  a.lse_acc = reinterpret_cast<float*>(ws + round_up(o_bytes, 256));
  a.partial_bf16 = plan->partial_bf16;
  a.out = out;
  a.out_dtype = out_dtype;
  a.inv_scale = out_inv_scale;
  a.lse_out = lse_out;
  a.sink = sink;
  a.amax = amax_out;
  a.status = dev->status;
  a.check_idx = g_check_idx.load();
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.drain_limit_ns = kWaitLimitNs;
  if ((st = cuda_status(skv::launch_mla_decode(tq, a, cs))) != MLA_OK) return st;
  const size_t out_esz = out_dtype == MLA_OUT_F32 ? 4 : (out_dtype == MLA_OUT_BF16 ? 2 : 1);
  skv::CombineArgs c{};
  c.o_acc = a.o_acc;
  c.lse_acc = a.lse_acc;
  c.partial_bf16 = a.partial_bf16;
  c.num_splits = tail_splits;
  c.rows = r * kMlaHeads;
  c.heads = kMlaHeads;
  c.d = kMlaDv;
  c.sink = sink;
  c.out = static_cast<uint8_t*>(out) + static_cast<size_t>(tail_first) * kMlaHeads * kMlaDv * out_esz;
  c.out_dtype = out_dtype;
  c.inv_scale = out_inv_scale;
  c.lse_out = lse_out != nullptr ? lse_out + static_cast<size_t>(tail_first) * kMlaHeads : nullptr;
  c.amax = amax_out;
  c.num_sms = dev->num_sms;
  return cuda_status(skv::launch_combine(c, /*zero_amax=*/false, /*pdl=*/true, cs));
}

// The one-shot call on the balanced schedule: every SM walks (nearly) the same
// number of 64-row blocks whatever s_q is. The decode kernel writes the final
// rows of whole tokens and a partial per piece of every token cut by a range
// boundary; the combine, launched as its programmatic dependent, folds those.
int mla_decode_balanced(const mla_plan_t* plan, int s_q, const void* q, const void* kv, int64_t n_kv,
                        const int32_t* idx, float sm_scale, const float* sink, int out_dtype, float out_inv_scale,
                        void* out, float* lse_out, float* amax_out, void* workspace, void* stream) {
  if (plan->h_q != kMlaHeads || plan->d_qk != kMlaDqk || plan->d_v != kMlaDv) return MLA_ERR_UNSUPPORTED;
  if (s_q > plan->s_q_max || plan->num_sms < 1 || plan->num_blocks < 1) return MLA_ERR_INVALID_ARG;
  int st = check_mla_inputs(s_q, plan->topk, q, kv, n_kv, idx, sm_scale);
  if (st != MLA_OK) return st;
  if (out == nullptr || !aligned(out, 16) || !valid_out_dtype(out_dtype)) return MLA_ERR_INVALID_ARG;
  if (out_dtype == MLA_OUT_E4M3 && !std::isfinite(out_inv_scale)) return MLA_ERR_INVALID_ARG;
  const int nb = plan->num_blocks;
  const int64_t U = static_cast<int64_t>(s_q) * nb;
  if (U > 0x7FFFFFFFll) return MLA_ERR_INVALID_ARG;
  const int P = balanced_ctas(s_q, nb, plan->num_sms);
  if (P > plan->balanced_ctas) return MLA_ERR_WORKSPACE;
  const int slots = balanced_slots(plan->s_q_max, nb, plan->num_sms);
  const int esz = plan->partial_bf16 ? 2 : 4;
  const uint64_t o_bytes = static_cast<uint64_t>(slots) * plan->s_q_max * kMlaHeads * kMlaDv * static_cast<uint64_t>(esz);
  if (workspace == nullptr || !aligned(workspace, 256) ||
      plan->workspace_bytes < split_workspace_bytes(slots, plan->s_q_max, esz))
    return MLA_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != MLA_OK) return st;
  CUtensorMap tq;
  if ((st = mla_q_tensor_map(s_q, q, &tq)) != MLA_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (amax_out != nullptr) {
    if ((st = cuda_status(cudaMemsetAsync(amax_out, 0, sizeof(float), cs))) != MLA_OK) return st;
  }
  skv::MlaArgs a{};
  a.kv = static_cast<const uint8_t*>(kv);
  a.idx = idx;
  a.s_q = s_q;
  a.topk = plan->topk;
  a.n_kv = static_cast<int>(n_kv);
  a.num_splits = 1;
  a.num_blocks = nb;
  a.dim_groups = 1;
  a.sched = 1;
  a.num_ctas = P;
  a.direct_whole = 1;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.o_acc = reinterpret_cast<float*>(ws);
  a.lse_acc = reinterpret_cast<float*>(ws + round_up(o_bytes, 256));
  a.partial_bf16 = plan->partial_bf16;
  a.out = out;
  a.out_dtype = out_dtype;
  a.inv_scale = out_inv_scale;
  a.lse_out = lse_out;
  a.sink = sink;
  a.amax = amax_out;
  a.status = dev->status;
  a.check_idx = g_check_idx.load();
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.drain_limit_ns = kWaitLimitNs;
  if ((st = cuda_status(skv::launch_mla_decode(tq, a, cs))) != MLA_OK) return st;
  skv::CombineArgs c{};
  c.o_acc = a.o_acc;
  c.lse_acc = a.lse_acc;
  c.partial_bf16 = a.partial_bf16;
  c.num_splits = slots;
  c.rows = s_q * kMlaHeads;
  c.heads = kMlaHeads;
  c.d = kMlaDv;
  c.sink = sink;
  c.out = out;
  c.out_dtype = out_dtype;
  c.inv_scale = out_inv_scale;
  c.lse_out = lse_out;
  c.amax = amax_out;
  c.num_sms = dev->num_sms;
  c.bal_nb = nb;
  c.bal_units = static_cast<int>(U);
  c.bal_ctas = P;
  return cuda_status(skv::launch_combine(c, /*zero_amax=*/false, /*pdl=*/true, cs));
}
}  // namespace

extern "C" {

int mla_workspace_init(const mla_plan_t* plan, void* workspace, void* stream) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARG;
  if (plan->workspace_bytes == 0) return MLA_OK;
  if (workspace == nullptr || !aligned(workspace, 256)) return MLA_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  const int st = device_state(&dev);
  if (st != MLA_OK) return st;
  return cuda_status(cudaMemsetAsync(workspace, 0, plan->workspace_bytes, static_cast<cudaStream_t>(stream)));
}

int mla_split_combine(const mla_plan_t* plan, int s_q, const void* workspace, const float* sink, int out_dtype,
                      float out_inv_scale, void* out, float* lse_out, float* amax_out, void* stream) {
  return mla_combine_impl(plan, s_q, workspace, sink, out_dtype, out_inv_scale, out, lse_out, amax_out, true,
                          stream);
}

}  // extern "C"

namespace {
// The unsplit launch with `dim_groups` CTAs per token (0: chosen from the
// device's SM count).
int mla_direct_impl(int s_q, int topk, const void* q, const void* kv, int64_t n_kv, const int32_t* idx,
                    float sm_scale, const float* sink, int out_dtype, float out_inv_scale, void* out, float* lse_out,
                    float* amax_out, int dim_groups, void* stream, int tail_first = 0, int tail_dgroups = 0) {
  int st = check_mla_inputs(s_q, topk, q, kv, n_kv, idx, sm_scale);
  if (st != MLA_OK) return st;
  if (out == nullptr || !aligned(out, 16) || !valid_out_dtype(out_dtype)) return MLA_ERR_INVALID_ARG;
  if (out_dtype == MLA_OUT_E4M3 && !std::isfinite(out_inv_scale)) return MLA_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != MLA_OK) return st;
  CUtensorMap tq;
  if ((st = mla_q_tensor_map(s_q, q, &tq)) != MLA_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (amax_out != nullptr) {
    if ((st = cuda_status(cudaMemsetAsync(amax_out, 0, sizeof(float), cs))) != MLA_OK) return st;
  }
  skv::MlaArgs a{};
  a.kv = static_cast<const uint8_t*>(kv);
  a.idx = idx;
  a.s_q = s_q;
  a.topk = topk;
  a.n_kv = static_cast<int>(n_kv);
  a.num_splits = 1;
  a.num_blocks = (topk + kMlaBlockRows - 1) / kMlaBlockRows;
  a.dim_groups = dim_groups > 0 ? dim_groups : dim_groups_for(s_q, dev->num_sms);
  a.sched = 0;
  a.direct_whole = 1;
  a.tail_first = tail_first;
  a.tail_dgroups = tail_dgroups;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.out = out;
  a.out_dtype = out_dtype;
  a.inv_scale = out_inv_scale;
  a.lse_out = lse_out;
  a.sink = sink;
  a.amax = amax_out;
  a.status = dev->status;
  a.check_idx = g_check_idx.load();
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.drain_limit_ns = kWaitLimitNs;
  return cuda_status(skv::launch_mla_decode(tq, a, cs));
}
}  // namespace

extern "C" {

int mla_sparse_decode_direct(int s_q, int topk, const void* q, const void* kv, int64_t n_kv, const int32_t* idx,
                             float sm_scale, const float* sink, int out_dtype, float out_inv_scale, void* out,
                             float* lse_out, float* amax_out, void* stream) {
  return mla_direct_impl(s_q, topk, q, kv, n_kv, idx, sm_scale, sink, out_dtype, out_inv_scale, out, lse_out,
                         amax_out, 0, stream);
}

int mla_sparse_decode(const mla_plan_t* plan, int s_q, const void* q, const void* kv, int64_t n_kv,
                      const int32_t* idx, float sm_scale, const float* sink, int out_dtype, float out_inv_scale,
                      void* out, float* lse_out, float* amax_out, void* workspace, void* stream) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARG;
  if (plan->balanced_ctas > 0 && plan->num_sms > 0 && plan->num_blocks > 0 && s_q >= 1 &&
      balanced_per(s_q, plan->num_blocks, plan->num_sms) > 0)
    return mla_decode_balanced(plan, s_q, q, kv, n_kv, idx, sm_scale, sink, out_dtype, out_inv_scale, out, lse_out,
                               amax_out, workspace, stream);
  int tail_first = 0, tail_splits = 0, tail_dgroups = 0;
  if (s_q >= 1 && s_q <= plan->s_q_max && tail_of(plan, s_q, &tail_first, &tail_splits, &tail_dgroups)) {
    if (tail_splits > 0)
      return mla_decode_tail(plan, s_q, q, kv, n_kv, idx, sm_scale, sink, out_dtype, out_inv_scale, out, lse_out,
                             amax_out, workspace, tail_first, tail_splits, stream);
    return mla_direct_impl(s_q, plan->topk, q, kv, n_kv, idx, sm_scale, sink, out_dtype, out_inv_scale, out,
                           lse_out, amax_out, 1, stream, tail_first, tail_dgroups);
  }
  if (plan->num_splits == 1) {
    if (s_q > plan->s_q_max) return MLA_ERR_INVALID_ARG;
    return mla_direct_impl(s_q, plan->topk, q, kv, n_kv, idx, sm_scale, sink, out_dtype, out_inv_scale, out,
                           lse_out, amax_out, plan->dim_groups, stream);
  }
  // validate the combine's own arguments before launching anything
  if (out == nullptr || !aligned(out, 16) || !valid_out_dtype(out_dtype)) return MLA_ERR_INVALID_ARG;
  if (out_dtype == MLA_OUT_E4M3 && !std::isfinite(out_inv_scale)) return MLA_ERR_INVALID_ARG;
  if (amax_out != nullptr &&
      cudaMemsetAsync(amax_out, 0, sizeof(float), static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  const int st = mla_sparse_decode_split(plan, s_q, q, kv, n_kv, idx, sm_scale, workspace, stream);
  if (st != MLA_OK) return st;
  return mla_combine_impl(plan, s_q, workspace, sink, out_dtype, out_inv_scale, out, lse_out, amax_out, false,
                          stream);
}

int mla_sparse_decode_host(const mla_plan_t* plan, int s_q, const void* q_host, void* q_dev, const void* kv,
                           int64_t n_kv, const int32_t* idx_host, int32_t* idx_dev, float sm_scale,
                           const float* sink, int out_dtype, float out_inv_scale, void* out_dev, void* out_host,
                           float* lse_dev, float* lse_host, float* amax_out, void* workspace, void* stream) {
  if (plan == nullptr || s_q < 1 || plan->topk < 1 || plan->h_q != kMlaHeads) return MLA_ERR_INVALID_ARG;
  if (q_host == nullptr || q_dev == nullptr || idx_host == nullptr || idx_dev == nullptr || out_dev == nullptr ||
      out_host == nullptr || (lse_dev == nullptr) != (lse_host == nullptr) || !valid_out_dtype(out_dtype))
    return MLA_ERR_INVALID_ARG;
  const size_t rows = static_cast<size_t>(s_q) * kMlaHeads;
  const size_t q_bytes = rows * kMlaDqk * 2;
  const size_t idx_bytes = static_cast<size_t>(s_q) * plan->topk * sizeof(int32_t);
  const size_t out_bytes = rows * kMlaDv * (out_dtype == MLA_OUT_F32 ? 4 : out_dtype == MLA_OUT_BF16 ? 2 : 1);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto copy = [&](void* dst, const void* src, size_t n, cudaMemcpyKind kind) {
    if (cudaMemcpyAsync(dst, src, n, kind, st) == cudaSuccess) return true;
    cudaGetLastError();
    return false;
  };
  if (!copy(q_dev, q_host, q_bytes, cudaMemcpyHostToDevice) ||
      !copy(idx_dev, idx_host, idx_bytes, cudaMemcpyHostToDevice))
    return MLA_ERR_CUDA;
  const int rc = mla_sparse_decode(plan, s_q, q_dev, kv, n_kv, idx_dev, sm_scale, sink, out_dtype, out_inv_scale,
                                   out_dev, lse_dev, amax_out, workspace, stream);
  if (rc != MLA_OK) return rc;
  if (!copy(out_host, out_dev, out_bytes, cudaMemcpyDeviceToHost)) return MLA_ERR_CUDA;
  if (lse_dev != nullptr && !copy(lse_host, lse_dev, rows * sizeof(float), cudaMemcpyDeviceToHost))
    return MLA_ERR_CUDA;
  return MLA_OK;
}

// ---------------------------------------------------------------- dense -----

int sdpa_fp8_decode_plan(int batch, int h_q, int h_kv, int d, int max_q_per_seq, int total_q_max, int max_kv,
                         int num_sms, int max_splits, int force_splits, sdpa_plan_t* out) {
  if (out == nullptr) return MLA_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  if (d != 128) return MLA_ERR_UNSUPPORTED;
  if (batch < 1 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0) return MLA_ERR_INVALID_ARG;
  const int group = h_q / h_kv;
  if (group > 64 || max_q_per_seq < 1 || group * max_q_per_seq > 64) return MLA_ERR_UNSUPPORTED;
  if (total_q_max < 1 || max_kv < 1 || num_sms < 0) return MLA_ERR_INVALID_ARG;
  if (max_splits < 0 || max_splits > MLA_MAX_SPLITS || force_splits < 0 || force_splits > MLA_MAX_SPLITS)
    return MLA_ERR_INVALID_ARG;
  if (num_sms == 0) {
    DeviceState* dv = nullptr;
    const int st = device_state(&dv);
    if (st != MLA_OK) return st;
    num_sms = dv->num_sms;
  }
  const int ntiles = (max_kv + 127) / 128;
  int S = force_splits;
  int adaptive = 0;
  if (S == 0) {
    // Each sequence gets its own split count, from the KV lengths, on the GPU:
    // the batch's tiles x KV heads are spread over one wave of SMs (T tiles per
    // split), so a ragged batch does not leave SMs idle behind its longest
    // sequence. S bounds the count (and sizes the workspace).
    const int cap = max_splits > 0 ? max_splits : MLA_MAX_SPLITS;
    S = std::min(std::min(cap, kDenseMaxAdaptiveSplits), ntiles);
    if (S < 1) S = 1;
    adaptive = S > 1 ? 1 : 0;
  }
  out->batch = batch;
  out->h_q = h_q;
  out->h_kv = h_kv;
  out->d = d;
  out->max_q_per_seq = max_q_per_seq;
  out->total_q_max = total_q_max;
  out->max_kv = max_kv;
  out->key_tile = 128;
  out->num_splits = S;
  out->num_sms = num_sms;
  out->adaptive_splits = adaptive;
  if (S > 1) {
    out->o_acc_bytes = static_cast<uint64_t>(S) * total_q_max * h_q * d * 4ull;
    out->lse_acc_offset = round_up(out->o_acc_bytes, 256);
    out->lse_acc_bytes = static_cast<uint64_t>(S) * total_q_max * h_q * 4ull;
    out->workspace_bytes = round_up(out->lse_acc_offset + out->lse_acc_bytes, 256);
  }
  return MLA_OK;
}

namespace {
int sdpa_launch(int batch, int h_q, int h_kv, int total_q, int64_t total_kv, int num_splits, const void* q,
                const void* k, const void* v, const int32_t* cu_q, const int32_t* cu_kv, const float* dq,
                const float* dk, const float* dv, float sm_scale, float* o_acc, float* lse_acc, void* out,
                int out_dtype, float inv_scale, float* lse_out, float* amax, bool direct, void* stream,
                int adaptive = 0, int num_sms = 0) {
  if (batch < 1 || h_kv < 1 || h_q < h_kv || h_q % h_kv != 0) return MLA_ERR_INVALID_ARG;
  if (adaptive && (direct || num_sms < 1)) return MLA_ERR_INVALID_ARG;
  const int group = h_q / h_kv;
  if (64 % group != 0) return MLA_ERR_UNSUPPORTED;
  if (q == nullptr || k == nullptr || v == nullptr || cu_q == nullptr || cu_kv == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(cu_q, 4) || !aligned(cu_kv, 4))
    return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale) || total_q < 1 || total_kv < 1 || total_kv > 0x7FFFFFFFll) return MLA_ERR_INVALID_ARG;
  if (num_splits < 1 || num_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(batch) * h_kv * num_splits > 0x7FFFFFFFll) return MLA_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  int st = device_state(&dev);
  if (st != MLA_OK) return st;
  CUtensorMap tq, tk, tv;
  {
    const uint64_t dims[3] = {128, static_cast<uint64_t>(h_q), static_cast<uint64_t>(total_q)};
    const uint64_t strides[2] = {128, static_cast<uint64_t>(h_q) * 128};
    const uint32_t box[3] = {128, static_cast<uint32_t>(group), static_cast<uint32_t>(64 / group)};
    if ((st = encode_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, dims, strides, box)) != MLA_OK) return st;
  }
  {
    const uint64_t dims[3] = {128, static_cast<uint64_t>(h_kv), static_cast<uint64_t>(total_kv)};
    const uint64_t strides[2] = {128, static_cast<uint64_t>(h_kv) * 128};
    const uint32_t box[3] = {128, 1, 128};
    if ((st = encode_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, k, dims, strides, box)) != MLA_OK) return st;
    if ((st = encode_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, v, dims, strides, box)) != MLA_OK) return st;
  }
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (direct && amax != nullptr) {
    if ((st = cuda_status(cudaMemsetAsync(amax, 0, sizeof(float), cs))) != MLA_OK) return st;
  }
  skv::SdpaArgs a{};
  a.q = static_cast<const uint8_t*>(q);
  a.cu_q = cu_q;
  a.cu_kv = cu_kv;
  a.descale_q = dq;
  a.descale_k = dk;
  a.descale_v = dv;
  a.batch = batch;
  a.h_q = h_q;
  a.h_kv = h_kv;
  a.total_q = total_q;
  a.num_splits = num_splits;
  a.adaptive = adaptive;
  a.num_sms = num_sms;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.o_acc = o_acc;
  a.lse_acc = lse_acc;
  a.out = out;
  a.out_dtype = out_dtype;
  a.inv_scale = inv_scale;
  a.lse_out = lse_out;
  a.amax = amax;
  a.status = dev->status;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.drain_limit_ns = kWaitLimitNs;
  return cuda_status(skv::launch_sdpa_decode(tq, tk, tv, a, direct, cs));
}
int sdpa_combine_impl(const sdpa_plan_t* plan, int total_q, const void* workspace, int out_dtype,
                      float out_inv_scale, void* out, float* lse_out, float* amax_out, bool zero_amax,
                      void* stream) {
  if (plan == nullptr || plan->num_splits < 2 || plan->num_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
  if (plan->d != 128) return MLA_ERR_UNSUPPORTED;
  if (total_q < 1 || total_q > plan->total_q_max || out == nullptr || !aligned(out, 16)) return MLA_ERR_INVALID_ARG;
  if (!valid_out_dtype(out_dtype)) return MLA_ERR_INVALID_ARG;
  if (out_dtype == MLA_OUT_E4M3 && !std::isfinite(out_inv_scale)) return MLA_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256) || plan->workspace_bytes == 0) return MLA_ERR_WORKSPACE;
  DeviceState* dev = nullptr;
  const int st = device_state(&dev);
  if (st != MLA_OK) return st;
  skv::CombineArgs c{};
  c.o_acc = static_cast<const float*>(workspace);
  c.lse_acc = reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) + plan->lse_acc_offset);
  c.num_splits = plan->num_splits;
  c.rows = total_q * plan->h_q;
  c.heads = plan->h_q;
  c.d = 128;
  c.sink = nullptr;
  c.out = out;
  c.out_dtype = out_dtype;
  c.inv_scale = out_inv_scale;
  c.lse_out = lse_out;
  c.amax = amax_out;
  c.num_sms = dev->num_sms;
  // per-sequence split counts: the slots past a sequence's own count hold LSE =
  // -inf and an O that was never written, so nothing is read before its weight
  c.sparse_splits = plan->adaptive_splits;
  return cuda_status(skv::launch_combine(c, zero_amax, /*pdl=*/true, static_cast<cudaStream_t>(stream)));
}

}  // namespace

int sdpa_fp8_decode_split(const sdpa_plan_t* plan, int total_q, int64_t total_kv, const void* q, const void* k,
                          const void* v, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                          const float* descale_q, const float* descale_k, const float* descale_v, float sm_scale,
                          void* workspace, void* stream) {
  if (plan == nullptr || plan->num_splits < 2 || plan->num_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
  if (plan->d != 128) return MLA_ERR_UNSUPPORTED;
  if (total_q < 1 || total_q > plan->total_q_max) return MLA_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256) || plan->workspace_bytes == 0) return MLA_ERR_WORKSPACE;
  return sdpa_launch(plan->batch, plan->h_q, plan->h_kv, total_q, total_kv, plan->num_splits, q, k, v,
                     cu_seqlens_q, cu_seqlens_kv, descale_q, descale_k, descale_v, sm_scale,
                     static_cast<float*>(workspace),
                     reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan->lse_acc_offset), nullptr, 0,
                     1.f, nullptr, nullptr, false, stream, plan->adaptive_splits, plan->num_sms);
}

int sdpa_split_combine(const sdpa_plan_t* plan, int total_q, const void* workspace, int out_dtype,
                       float out_inv_scale, void* out, float* lse_out, float* amax_out, void* stream) {
  return sdpa_combine_impl(plan, total_q, workspace, out_dtype, out_inv_scale, out, lse_out, amax_out, true, stream);
}

int sdpa_fp8_decode_direct(int batch, int h_q, int h_kv, int d, int total_q, int64_t total_kv, const void* q,
                           const void* k, const void* v, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                           const float* descale_q, const float* descale_k, const float* descale_v, float sm_scale,
                           int out_dtype, float out_inv_scale, void* out, float* lse_out, float* amax_out,
                           void* stream) {
  if (d != 128) return MLA_ERR_UNSUPPORTED;
  if (out == nullptr || !aligned(out, 16) || !valid_out_dtype(out_dtype)) return MLA_ERR_INVALID_ARG;
  if (out_dtype == MLA_OUT_E4M3 && !std::isfinite(out_inv_scale)) return MLA_ERR_INVALID_ARG;
  return sdpa_launch(batch, h_q, h_kv, total_q, total_kv, 1, q, k, v, cu_seqlens_q, cu_seqlens_kv, descale_q,
                     descale_k, descale_v, sm_scale, nullptr, nullptr, out, out_dtype, out_inv_scale, lse_out,
                     amax_out, true, stream);
}

int sdpa_fp8_decode(const sdpa_plan_t* plan, int total_q, int64_t total_kv, const void* q, const void* k,
                    const void* v, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                    const float* descale_q, const float* descale_k, const float* descale_v, float sm_scale,
                    int out_dtype, float out_inv_scale, void* out, float* lse_out, float* amax_out,
                    void* workspace, void* stream) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARG;
  if (total_q > plan->total_q_max) return MLA_ERR_INVALID_ARG;
  if (plan->num_splits == 1)
    return sdpa_fp8_decode_direct(plan->batch, plan->h_q, plan->h_kv, plan->d, total_q, total_kv, q, k, v,
                                  cu_seqlens_q, cu_seqlens_kv, descale_q, descale_k, descale_v, sm_scale, out_dtype,
                                  out_inv_scale, out, lse_out, amax_out, stream);
  if (out == nullptr || !aligned(out, 16) || !valid_out_dtype(out_dtype)) return MLA_ERR_INVALID_ARG;
  if (out_dtype == MLA_OUT_E4M3 && !std::isfinite(out_inv_scale)) return MLA_ERR_INVALID_ARG;
  if (amax_out != nullptr &&
      cudaMemsetAsync(amax_out, 0, sizeof(float), static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  const int st = sdpa_fp8_decode_split(plan, total_q, total_kv, q, k, v, cu_seqlens_q, cu_seqlens_kv, descale_q,
                                       descale_k, descale_v, sm_scale, workspace, stream);
  if (st != MLA_OK) return st;
  return sdpa_combine_impl(plan, total_q, workspace, out_dtype, out_inv_scale, out, lse_out, amax_out, false,
                           stream);
}

// ---------------------------------------------------------------- status ----

int mla_get_status(uint32_t* status_out, uint32_t* site_out) {
  DeviceState* dev = nullptr;
  const int st = device_state(&dev);
  if (st != MLA_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  uint32_t h[2] = {0, 0};
  if (cudaMemcpy(h, dev->status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  const uint32_t zero[2] = {0, 0};
  if (cudaMemcpy(dev->status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  if (status_out != nullptr) *status_out = h[0];
  if (site_out != nullptr) *site_out = h[1];
  return MLA_OK;
}

int mla_set_wait_limit_ns(uint64_t limit_ns) {
  if (limit_ns == 0) limit_ns = kWaitLimitNs;
  if (limit_ns < 100ull || limit_ns > 10000000000ull) return MLA_ERR_INVALID_ARG;
  g_wait_limit_ns.store(limit_ns);
  return MLA_OK;
}

int mla_set_index_checks(int enable) {
  if (enable != 0 && enable != 1) return MLA_ERR_INVALID_ARG;
  g_check_idx.store(enable);
  return MLA_OK;
}

int mla_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  DeviceState* dev = nullptr;
  const int st = device_state(&dev);
  if (st != MLA_OK) return st;
  if (limit_ns == 0 || limit_ns > 10000000000ull) return MLA_ERR_INVALID_ARG;
  return cuda_status(skv::launch_wait_selftest(dev->status, limit_ns, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ------------------------------------------------------- no-allocation entry --
//
// A decode call for callers that cannot allocate device memory: the partial
// workspace of the split pass lives in this file-scope array instead of a
// caller buffer. The array is part of the library's device image, so every GPU
// that loads the library holds MLA_NOALLOC_SCRATCH_BYTES of it until the
// process exits.
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};   // device address of g_noalloc_scratch, per device

// Resolves the array's device address for the current device (once per device,
// with that device current). In host code the symbol itself is only a stand-in,
// never a device address, so it must not be handed to a kernel.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MLA_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_sparse_decode_noalloc(int s_q, int topk, const void* q, const void* kv, int64_t n_kv, const int32_t* idx,
                              float sm_scale, const float* sink, int num_splits, int out_dtype, float out_inv_scale,
                              void* out, float* lse_out, float* amax_out, void* stream) {
  if (num_splits < 0 || num_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
  if (s_q < 1) return MLA_ERR_INVALID_ARG;
  // The automatic choice only considers split counts whose workspace fits the
  // array, so it never refuses an ordinary shape; a forced count is taken as
  // asked and refused below if it does not fit.
  int max_splits = 0;
  if (num_splits == 0) {
    max_splits = 1;
    for (int S = 2; S <= MLA_MAX_SPLITS; ++S)
      if (split_workspace_bytes(S, s_q) <= MLA_NOALLOC_SCRATCH_BYTES) max_splits = S;
  }
  mla_plan_t plan;
  int st = mla_decode_plan(s_q, kMlaHeads, kMlaDqk, kMlaDv, topk, 0, max_splits, num_splits, &plan);
  if (st != MLA_OK) return st;
  // the (token, split) jobs: their workspace is num_splits * s_q partial rows
  plan.balanced_ctas = 0;
  plan.tail_ctas = 0;
  plan.workspace_bytes = plan.num_splits > 1 ? round_up(plan.lse_acc_offset + plan.lse_acc_bytes, 256) : 0;
  if (plan.workspace_bytes > MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (plan.workspace_bytes > 0 && (st = noalloc_scratch(&scratch)) != MLA_OK) return st;
  // Same split + combine (or direct) launches as mla_sparse_decode; the split
  // pass writes every partial slot it owns before the combine reads it, so
  // nothing in the scratch array needs to start at zero.
  return mla_sparse_decode(&plan, s_q, q, kv, n_kv, idx, sm_scale, sink, out_dtype, out_inv_scale, out, lse_out,
                           amax_out, scratch, stream);
}

}  // extern "C"

// C-ABI entry points: host-side validation, launch
// planning (head-group width, persistent grid size and schedule) and
// launches on the caller's stream.  See include/sparse_mla.h for the contract of each call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "bwd_kernel.cuh"
#include "fwd_kernel.cuh"
#include "indexer_kernel.cuh"
#include "sparse_mla.h"

namespace {

using smla::FwdParams;

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 1000000000ull;
std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};

struct DeviceState {
  bool probed = false;
  bool supported = false;
  int sm_count = 0;
  bool attrs_set = false;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Top-k kernel: histogram and the staged keys of a row of up to
// kTopkStageCap positions.
constexpr int kTopkStageCap = 49152;
constexpr int kTopkMaxSmem = smla::kTopkBins * 4 + kTopkStageCap * 4;

sparse_mla_status_t device_setup(int* sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPARSE_MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SPARSE_MLA_ERR_CUDA;
    st.supported = (major == 10 && minor == 3);
    st.sm_count = sms;
    st.probed = true;
  }
  if (!st.supported) return SPARSE_MLA_ERR_UNSUPPORTED_ARCH;
  if (!st.attrs_set) {
    if (cudaFuncSetAttribute(smla::sparse_mla_fwd_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smla::smem_bytes<16>()) != cudaSuccess ||
        cudaFuncSetAttribute(smla::sparse_mla_fwd_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smla::smem_bytes<32>()) != cudaSuccess ||
        cudaFuncSetAttribute(smla::sparse_mla_fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smla::smem_bytes<64>()) != cudaSuccess ||
        cudaFuncSetAttribute(smla::sparse_mla_fwd_kernel<16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smla::smem_bytes<16, true>()) != cudaSuccess ||
        cudaFuncSetAttribute(smla::sparse_mla_fwd_kernel<32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smla::smem_bytes<32>()) != cudaSuccess ||
        cudaFuncSetAttribute(smla::sparse_mla_fwd_kernel<64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smla::smem_bytes<64>()) != cudaSuccess ||
        cudaFuncSetAttribute(smla::sparse_mla_bwd_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smla::bwd_smem_bytes<1>()) != cudaSuccess ||
        cudaFuncSetAttribute(smla::sparse_mla_bwd_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smla::bwd_smem_bytes<2>()) != cudaSuccess ||
        cudaFuncSetAttribute(smla::dsa_scores_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smla::idx_smem_bytes()) != cudaSuccess ||
        cudaFuncSetAttribute(smla::dsa_scores_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smla::idx_smem_bytes()) != cudaSuccess ||
        cudaFuncSetAttribute(smla::dsa_scores_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smla::idx_smem_bytes()) != cudaSuccess ||
        cudaFuncSetAttribute(smla::dsa_topk_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTopkMaxSmem) != cudaSuccess ||
        cudaFuncSetAttribute(smla::dsa_topk_kernel<1024>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTopkMaxSmem) != cudaSuccess)
      return SPARSE_MLA_ERR_CUDA;
    st.attrs_set = true;
  }
  *sm_count = st.sm_count;
  return SPARSE_MLA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Head-group width N (the MMA's N): 16, 32 or 64; more heads use several
// 64-wide groups (one CTA per group).
int head_width(int h_q) { return h_q <= 16 ? 16 : (h_q <= 32 ? 32 : 64); }
int head_groups(int h_q) { return (h_q + 63) / 64; }

// Persistent grids: each CTA takes ~225 KB of shared memory, so one runs per
// SM, and every CTA works through a list of items (see Sched in the kernel).
int blocks_per_list(int topk) { return (topk + smla::kBlk - 1) / smla::kBlk; }

// Prefill: whole units (token x head group) over min(units, SMs) CTAs.
int prefill_ctas(long long n_tok, int h_q, int sm_count) {
  const long long units = n_tok * head_groups(h_q);
  return static_cast<int>(units < sm_count ? units : sm_count);
}

// Decode: the units' block lists laid end to end and cut into equal ranges,
// one per CTA, at most one CTA per SM.  Every range holds at least
// ceil(nb / 31) blocks, so no unit is cut into more than 32 pieces (the
// merge keeps one piece per lane of a warp).
int decode_ctas(long long n_tok, int h_q, int topk, int sm_count) {
  const int nb = blocks_per_list(topk);
  const long long total = n_tok * head_groups(h_q) * nb;
  const long long min_blocks = (nb + 30) / 31;
  long long g = total / min_blocks;
  if (g > sm_count) g = sm_count;
  return static_cast<int>(g < 1 ? 1 : g);
}

// Head rows of one partial slot (a slot holds one unit's heads).
int part_rows(int h_q) { return h_q < 64 ? h_q : 64; }

// Decode workspace: partial outputs [2 G][part_rows][d_v] fp32, then partial
// LSEs [2 G][part_rows] (two slots per CTA: its first and last item).
size_t decode_part_floats(int ctas, int h_q) {
  return 2 * static_cast<size_t>(ctas) * static_cast<size_t>(part_rows(h_q)) * (static_cast<size_t>(smla::kDv) + 1);
}

// Decode workspace: the partials, then (16-byte aligned) one merge counter
// per (unit, softmax group), units = tokens x 64-head groups.
size_t decode_counter_offset(int ctas, int h_q) { return (decode_part_floats(ctas, h_q) * sizeof(float) + 15) & ~size_t(15); }
size_t decode_counter_bytes(long long n_tok, int h_q) {
  return static_cast<size_t>(n_tok) * static_cast<size_t>(head_groups(h_q)) * 2 * sizeof(int32_t);
}

// The forward grid (one persistent CTA per SM or fewer).
template <int N, bool kFp8>
cudaError_t launch_fwd_n(const FwdParams& p, cudaStream_t stream) {
  smla::sparse_mla_fwd_kernel<N, kFp8><<<dim3(static_cast<unsigned>(p.ctas)), smla::fwd_threads<N, kFp8>(),
                                         smla::smem_bytes<N, kFp8>(), stream>>>(p);
  return cudaGetLastError();
}

sparse_mla_status_t launch_fwd(const FwdParams& p, cudaStream_t stream) {
  const int N = head_width(p.h_q);
  const bool fp8 = p.mode == smla::kPagedFp8;
  cudaError_t e;
  if (N == 16) e = fp8 ? launch_fwd_n<16, true>(p, stream) : launch_fwd_n<16, false>(p, stream);
  else if (N == 32) e = fp8 ? launch_fwd_n<32, true>(p, stream) : launch_fwd_n<32, false>(p, stream);
  else e = fp8 ? launch_fwd_n<64, true>(p, stream) : launch_fwd_n<64, false>(p, stream);
  return e == cudaSuccess ? SPARSE_MLA_OK : SPARSE_MLA_ERR_CUDA;
}

sparse_mla_status_t launch_fill(void* out, float* lse, long long n_th, cudaStream_t stream) {
  if (n_th <= 0) return SPARSE_MLA_OK;
  const long long blocks = (n_th + 255) / 256;
  smla::fill_masked_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(
      static_cast<__nv_bfloat16*>(out), lse, n_th);
  return cudaGetLastError() == cudaSuccess ? SPARSE_MLA_OK : SPARSE_MLA_ERR_CUDA;
}

FwdParams base_params(const void* q, const int32_t* indices, float sm_scale, void* out, float* lse, int n_tok,
                      int h_q, int topk) {
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.indices = indices;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.n_tok = n_tok;
  p.h_q = h_q;
  p.topk = topk;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.sm_scale = sm_scale;
  p.groups = head_groups(h_q);
  p.nb = blocks_per_list(topk);
  p.part_rows = part_rows(h_q);
  unsigned long long t = g_timeout_ns.load();
  p.timeout_ns = t ? t : kDefaultTimeoutNs;
  return p;
}

sparse_mla_status_t check_common(const void* q, const int32_t* indices, const void* out, const float* lse,
                                 long long n_tok, int h_q, int d_qk, int d_v, int topk, bool need_indices = true) {
  if (n_tok < 0 || h_q < 1 || topk < 1) return SPARSE_MLA_ERR_INVALID_ARG;
  if (d_qk != smla::kDqk || d_v != smla::kDv) return SPARSE_MLA_ERR_UNSUPPORTED_SHAPE;
  if (n_tok > INT_MAX / 2 || static_cast<long long>(h_q) * 64 > INT_MAX) return SPARSE_MLA_ERR_INVALID_ARG;
  if (n_tok == 0) return SPARSE_MLA_OK;
  if (!q || (need_indices && !indices) || !out || !lse) return SPARSE_MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || (need_indices && !aligned(indices, 4)) || !aligned(lse, 4))
    return SPARSE_MLA_ERR_INVALID_ARG;
  return SPARSE_MLA_OK;
}

}  // namespace

extern "C" {

sparse_mla_status_t sparse_mla_fwd(const void* q, const void* kv, const int32_t* indices, float sm_scale, void* out,
                                   float* lse, int s_q, int s_kv, int h_q, int d_qk, int d_v, int topk,
                                   void* stream) {
  sparse_mla_status_t st = check_common(q, indices, out, lse, s_q, h_q, d_qk, d_v, topk);
  if (st != SPARSE_MLA_OK) return st;
  if (s_kv < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_setup(&sms)) != SPARSE_MLA_OK) return st;
  if (s_q == 0) return SPARSE_MLA_OK;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (s_kv == 0) return launch_fill(out, lse, static_cast<long long>(s_q) * h_q, cs);
  if (!kv || !aligned(kv, 16)) return SPARSE_MLA_ERR_INVALID_ARG;
  FwdParams p = base_params(q, indices, sm_scale, out, lse, s_q, h_q, topk);
  p.kv = static_cast<const __nv_bfloat16*>(kv);
  p.mode = smla::kDense;
  p.n_rows = s_kv;
  p.s_kv = s_kv;
  p.sched = smla::kWholeUnits;
  p.ctas = prefill_ctas(s_q, h_q, sms);
  return launch_fwd(p, cs);
}

sparse_mla_status_t sparse_mla_fwd_varlen(const void* q, const void* kv, const int32_t* indices,
                                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch,
                                          float sm_scale, void* out, float* lse, int total_q, int total_kv,
                                          int h_q, int d_qk, int d_v, int topk, void* stream) {
  sparse_mla_status_t st = check_common(q, indices, out, lse, total_q, h_q, d_qk, d_v, topk);
  if (st != SPARSE_MLA_OK) return st;
  if (total_kv < 0 || batch < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  if (total_q > 0 && (batch < 1 || !cu_seqlens_q || !cu_seqlens_kv || !aligned(cu_seqlens_q, 4) ||
                      !aligned(cu_seqlens_kv, 4)))
    return SPARSE_MLA_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_setup(&sms)) != SPARSE_MLA_OK) return st;
  if (total_q == 0) return SPARSE_MLA_OK;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (total_kv == 0) return launch_fill(out, lse, static_cast<long long>(total_q) * h_q, cs);
  if (!kv || !aligned(kv, 16)) return SPARSE_MLA_ERR_INVALID_ARG;
  FwdParams p = base_params(q, indices, sm_scale, out, lse, total_q, h_q, topk);
  p.kv = static_cast<const __nv_bfloat16*>(kv);
  p.mode = smla::kVarlen;
  p.n_rows = total_kv;
  p.batch = batch;
  p.cu_q = cu_seqlens_q;
  p.cu_kv = cu_seqlens_kv;
  p.sched = smla::kWholeUnits;
  p.ctas = prefill_ctas(total_q, h_q, sms);
  return launch_fwd(p, cs);
}

sparse_mla_status_t sparse_mla_fwd_causal(const void* q, const void* kv, float sm_scale, void* out, float* lse,
                                          int s_q, int s_kv, int h_q, int d_qk, int d_v, void* stream) {
  if (s_kv < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  // A token's list holds every KV position: topk = s_kv (at least 1 for the
  // shape checks; s_kv = 0 is the all-masked case below).
  sparse_mla_status_t st = check_common(q, nullptr, out, lse, s_q, h_q, d_qk, d_v, s_kv > 0 ? s_kv : 1, false);
  if (st != SPARSE_MLA_OK) return st;
  int sms = 0;
  if ((st = device_setup(&sms)) != SPARSE_MLA_OK) return st;
  if (s_q == 0) return SPARSE_MLA_OK;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (s_kv == 0) return launch_fill(out, lse, static_cast<long long>(s_q) * h_q, cs);
  if (!kv || !aligned(kv, 16)) return SPARSE_MLA_ERR_INVALID_ARG;
  FwdParams p = base_params(q, nullptr, sm_scale, out, lse, s_q, h_q, s_kv);
  p.kv = static_cast<const __nv_bfloat16*>(kv);
  p.mode = smla::kCausal;
  p.n_rows = s_kv;
  p.s_kv = s_kv;
  p.causal_off = s_kv - s_q;
  p.sched = smla::kWholeUnits;
  p.ctas = prefill_ctas(s_q, h_q, sms);
  return launch_fwd(p, cs);
}

}  // extern "C"

namespace {

// Shared tail of the two backward entry points: dkv zeroed on the stream,
// then the persistent backward grid over units of one token x 16 heads (x 32
// heads above 16).
sparse_mla_status_t launch_bwd(FwdParams p, long long n_tok, int h_q, long long n_rows, float* dq, float* dkv,
                               int sms, cudaStream_t cs) {
  if (n_rows > 0 &&
      cudaMemsetAsync(dkv, 0, static_cast<size_t>(n_rows) * smla::kDqk * sizeof(float), cs) != cudaSuccess)
    return SPARSE_MLA_ERR_CUDA;
  if (n_tok == 0) return SPARSE_MLA_OK;
  if (n_rows == 0)
    return cudaMemsetAsync(dq, 0, static_cast<size_t>(n_tok) * h_q * smla::kDqk * sizeof(float), cs) ==
                   cudaSuccess
               ? SPARSE_MLA_OK
               : SPARSE_MLA_ERR_CUDA;
  p.dq = dq;
  p.dkv = dkv;
  // Units of 16 heads up to 16 heads, else of 32 (two halves of 16 that
  // share the gather and each block's dkv reduction).
  const int unit_heads = h_q <= smla::kBwdHeads ? smla::kBwdHeads : 2 * smla::kBwdHeads;
  p.groups = (h_q + unit_heads - 1) / unit_heads;
  p.sched = smla::kWholeUnits;
  const long long units = n_tok * p.groups;
  p.ctas = static_cast<int>(units < sms ? units : sms);
  if (unit_heads == smla::kBwdHeads)
    smla::sparse_mla_bwd_kernel<1><<<p.ctas, smla::BwdLayout<1>::kThreads, smla::bwd_smem_bytes<1>(), cs>>>(p);
  else
    smla::sparse_mla_bwd_kernel<2><<<p.ctas, smla::BwdLayout<2>::kThreads, smla::bwd_smem_bytes<2>(), cs>>>(p);
  return cudaGetLastError() == cudaSuccess ? SPARSE_MLA_OK : SPARSE_MLA_ERR_CUDA;
}

sparse_mla_status_t check_bwd(const void* dout, const float* dq, const float* dkv, long long n_tok,
                              long long n_rows) {
  if (n_tok > 0 && (!dout || !dq || !aligned(dout, 16) || !aligned(dq, 16))) return SPARSE_MLA_ERR_INVALID_ARG;
  if (n_rows > 0 && (!dkv || !aligned(dkv, 16))) return SPARSE_MLA_ERR_INVALID_ARG;
  return SPARSE_MLA_OK;
}

}  // namespace

extern "C" {

sparse_mla_status_t sparse_mla_bwd(const void* q, const void* kv, const int32_t* indices, const void* out,
                                   const float* lse, const void* dout, float sm_scale, float* dq, float* dkv,
                                   int s_q, int s_kv, int h_q, int d_qk, int d_v, int topk, void* stream) {
  sparse_mla_status_t st = check_common(q, indices, out, lse, s_q, h_q, d_qk, d_v, topk);
  if (st != SPARSE_MLA_OK) return st;
  if (s_kv < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  if ((st = check_bwd(dout, dq, dkv, s_q, s_kv)) != SPARSE_MLA_OK) return st;
  int sms = 0;
  if ((st = device_setup(&sms)) != SPARSE_MLA_OK) return st;
  if (s_q > 0 && s_kv > 0 && (!kv || !aligned(kv, 16))) return SPARSE_MLA_ERR_INVALID_ARG;
  FwdParams p = base_params(q, indices, sm_scale, const_cast<void*>(out), const_cast<float*>(lse), s_q, h_q, topk);
  p.kv = static_cast<const __nv_bfloat16*>(kv);
  p.mode = smla::kDense;
  p.n_rows = s_kv;
  p.s_kv = s_kv;
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  return launch_bwd(p, s_q, h_q, s_kv, dq, dkv, sms, static_cast<cudaStream_t>(stream));
}

sparse_mla_status_t sparse_mla_bwd_varlen(const void* q, const void* kv, const int32_t* indices,
                                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch,
                                          const void* out, const float* lse, const void* dout, float sm_scale,
                                          float* dq, float* dkv, int total_q, int total_kv, int h_q, int d_qk,
                                          int d_v, int topk, void* stream) {
  sparse_mla_status_t st = check_common(q, indices, out, lse, total_q, h_q, d_qk, d_v, topk);
  if (st != SPARSE_MLA_OK) return st;
  if (total_kv < 0 || batch < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  if (total_q > 0 && (batch < 1 || !cu_seqlens_q || !cu_seqlens_kv || !aligned(cu_seqlens_q, 4) ||
                      !aligned(cu_seqlens_kv, 4)))
    return SPARSE_MLA_ERR_INVALID_ARG;
  if ((st = check_bwd(dout, dq, dkv, total_q, total_kv)) != SPARSE_MLA_OK) return st;
  int sms = 0;
  if ((st = device_setup(&sms)) != SPARSE_MLA_OK) return st;
  if (total_q > 0 && total_kv > 0 && (!kv || !aligned(kv, 16))) return SPARSE_MLA_ERR_INVALID_ARG;
  FwdParams p = base_params(q, indices, sm_scale, const_cast<void*>(out), const_cast<float*>(lse), total_q, h_q,
                            topk);
  p.kv = static_cast<const __nv_bfloat16*>(kv);
  p.mode = smla::kVarlen;
  p.n_rows = total_kv;
  p.batch = batch;
  p.cu_q = cu_seqlens_q;
  p.cu_kv = cu_seqlens_kv;
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  return launch_bwd(p, total_q, h_q, total_kv, dq, dkv, sms, static_cast<cudaStream_t>(stream));
}

size_t sparse_mla_decode_workspace_size(int batch, int s_next, int h_q, int d_v, int topk) {
  if (batch < 1 || s_next < 1 || h_q < 1 || topk < 1 || d_v != smla::kDv) return 0;
  int sms = 0;
  if (device_setup(&sms) != SPARSE_MLA_OK) return 0;
  const long long n_tok = static_cast<long long>(batch) * s_next;
  const int ctas = decode_ctas(n_tok, h_q, topk, sms);
  if (ctas <= 1) return 0;   // one CTA runs every unit whole
  return decode_counter_offset(ctas, h_q) + decode_counter_bytes(n_tok, h_q);
}

}  // extern "C"

namespace {

// Argument checks of the paged decode (every decode entry point runs them
// first, in this order).  On OK, *sms holds the device's SM count.
sparse_mla_status_t check_decode(const void* q, const void* kv_cache, const int32_t* block_table,
                                 const int32_t* cache_seqlens, const int32_t* indices, const void* out,
                                 const float* lse, int batch, int s_next, int h_q, int d_qk, int d_v, int topk,
                                 int page_size, int max_blocks, int num_blocks, int* sms) {
  if (batch < 0 || s_next < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  const long long n_tok = static_cast<long long>(batch) * s_next;
  sparse_mla_status_t st = check_common(q, indices, out, lse, n_tok, h_q, d_qk, d_v, topk);
  if (st != SPARSE_MLA_OK) return st;
  if (page_size < 1 || max_blocks < 0 || num_blocks < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  if (static_cast<long long>(num_blocks) * page_size > INT_MAX) return SPARSE_MLA_ERR_INVALID_ARG;
  if (n_tok > 0 && (!block_table || !cache_seqlens || !aligned(block_table, 4) || !aligned(cache_seqlens, 4)))
    return SPARSE_MLA_ERR_INVALID_ARG;
  if ((st = device_setup(sms)) != SPARSE_MLA_OK) return st;
  if (n_tok == 0 || num_blocks == 0 || max_blocks == 0) return SPARSE_MLA_OK;
  if (!kv_cache || !aligned(kv_cache, 16)) return SPARSE_MLA_ERR_INVALID_ARG;
  // The kernel forms c * (units x blocks) in 64 bits for c up to the grid size.
  if (n_tok * head_groups(h_q) * blocks_per_list(topk) > (1LL << 62) / (*sms > 0 ? *sms : 1))
    return SPARSE_MLA_ERR_INVALID_ARG;
  return SPARSE_MLA_OK;
}

}  // namespace

extern "C" {

}  // extern "C"

namespace {

// The paged decode launch of both cache formats (mode kPaged or kPagedFp8):
// the forward grid over block ranges, then the merge of cut units.
sparse_mla_status_t run_decode(int mode, const void* q, const void* kv_cache, const int32_t* block_table,
                               const int32_t* cache_seqlens, const int32_t* indices, float sm_scale, void* out,
                               float* lse, int batch, int s_next, int h_q, int d_qk, int d_v, int topk,
                               int page_size, int max_blocks, int num_blocks, void* workspace,
                               size_t workspace_bytes, void* stream) {
  int sms = 0;
  sparse_mla_status_t st = check_decode(q, kv_cache, block_table, cache_seqlens, indices, out, lse, batch, s_next,
                                        h_q, d_qk, d_v, topk, page_size, max_blocks, num_blocks, &sms);
  if (st != SPARSE_MLA_OK) return st;
  const long long n_tok = static_cast<long long>(batch) * s_next;
  if (n_tok == 0) return SPARSE_MLA_OK;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (num_blocks == 0 || max_blocks == 0) return launch_fill(out, lse, n_tok * h_q, cs);
  const int ctas = decode_ctas(n_tok, h_q, topk, sms);
  const size_t need = sparse_mla_decode_workspace_size(batch, s_next, h_q, d_v, topk);
  if (need > 0 && (workspace_bytes < need || !workspace)) return SPARSE_MLA_ERR_WORKSPACE_TOO_SMALL;
  if (need > 0 && !aligned(workspace, 16)) return SPARSE_MLA_ERR_INVALID_ARG;
  FwdParams p = base_params(q, indices, sm_scale, out, lse, static_cast<int>(n_tok), h_q, topk);
  p.kv = static_cast<const __nv_bfloat16*>(kv_cache);   // kPagedFp8: read as bytes
  p.mode = mode;
  p.n_rows = num_blocks * page_size;
  p.batch = batch;
  p.s_next = s_next;
  p.page_size = page_size;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  p.block_table = block_table;
  p.seqlens = cache_seqlens;
  p.sched = smla::kBlockRanges;
  p.ctas = ctas;
  if (need > 0) {
    float* ws = static_cast<float*>(workspace);
    p.part_o = ws;
    p.part_lse = ws + 2 * static_cast<size_t>(ctas) * p.part_rows * smla::kDv;
    // Units cut between CTAs leave a partial per piece; the CTA that writes
    // a unit's last piece (counted here, from zero) merges them.
    p.merge_count = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) + decode_counter_offset(ctas, h_q));
    if (cudaMemsetAsync(p.merge_count, 0, decode_counter_bytes(n_tok, h_q), cs) != cudaSuccess)
      return SPARSE_MLA_ERR_CUDA;
  }
  return launch_fwd(p, cs);
}

}  // namespace

extern "C" {

sparse_mla_status_t sparse_mla_decode(const void* q, const void* kv_cache, const int32_t* block_table,
                                      const int32_t* cache_seqlens, const int32_t* indices, float sm_scale, void* out,
                                      float* lse, int batch, int s_next, int h_q, int d_qk, int d_v, int topk,
                                      int page_size, int max_blocks, int num_blocks, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  return run_decode(smla::kPaged, q, kv_cache, block_table, cache_seqlens, indices, sm_scale, out, lse, batch,
                    s_next, h_q, d_qk, d_v, topk, page_size, max_blocks, num_blocks, workspace, workspace_bytes,
                    stream);
}

sparse_mla_status_t sparse_mla_decode_fp8(const void* q, const void* kv_cache, const int32_t* block_table,
                                          const int32_t* cache_seqlens, const int32_t* indices, float sm_scale,
                                          void* out, float* lse, int batch, int s_next, int h_q, int d_qk, int d_v,
                                          int topk, int page_size, int max_blocks, int num_blocks, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  // Slots are 656 bytes: the pool's byte size must fit the 64-bit offsets the
  // gather forms (num_blocks * page_size fits int32, as for the bf16 cache).
  return run_decode(smla::kPagedFp8, q, kv_cache, block_table, cache_seqlens, indices, sm_scale, out, lse, batch,
                    s_next, h_q, d_qk, d_v, topk, page_size, max_blocks, num_blocks, workspace, workspace_bytes,
                    stream);
}

}  // extern "C"

namespace {

// Scratch of sparse_mla_decode_noalloc: a file-scope device array, so the
// entry point needs no allocation.  Every GPU that loads this library holds
// it until the process exits.  In host code the symbol is only a host-side
// stand-in; its device address comes from cudaGetSymbolAddress, taken once
// per device with that device current.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
void* g_noalloc_ptr[kMaxDevices] = {};

sparse_mla_status_t noalloc_scratch(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPARSE_MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SPARSE_MLA_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return SPARSE_MLA_OK;
}

}  // namespace

extern "C" {

size_t sparse_mla_decode_noalloc_max_scratch_bytes(void) { return kNoAllocScratchBytes; }

sparse_mla_status_t sparse_mla_decode_noalloc(const void* q, const void* kv_cache, const int32_t* block_table,
                                              const int32_t* cache_seqlens, const int32_t* indices, float sm_scale,
                                              void* out, float* lse, int batch, int s_next, int h_q, int d_qk,
                                              int d_v, int topk, int page_size, int max_blocks, int num_blocks,
                                              void* stream) {
  // The same argument checks as sparse_mla_decode, then the scratch size.
  int sms = 0;
  sparse_mla_status_t cst = check_decode(q, kv_cache, block_table, cache_seqlens, indices, out, lse, batch, s_next,
                                         h_q, d_qk, d_v, topk, page_size, max_blocks, num_blocks, &sms);
  if (cst != SPARSE_MLA_OK) return cst;
  const size_t need = sparse_mla_decode_workspace_size(batch, s_next, h_q, d_v, topk);
  if (need > kNoAllocScratchBytes) return SPARSE_MLA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  if (need > 0) {
    sparse_mla_status_t st = noalloc_scratch(&ws);
    if (st != SPARSE_MLA_OK) return st;
  }
  return sparse_mla_decode(q, kv_cache, block_table, cache_seqlens, indices, sm_scale, out, lse, batch, s_next,
                           h_q, d_qk, d_v, topk, page_size, max_blocks, num_blocks, ws,
                           need > 0 ? kNoAllocScratchBytes : 0, stream);
}

}  // extern "C"

namespace {

sparse_mla_status_t launch_valid_count(FwdParams& p, int32_t* counts, cudaStream_t cs) {
  if (cudaMemsetAsync(counts, 0, static_cast<size_t>(p.n_tok) * sizeof(int32_t), cs) != cudaSuccess)
    return SPARSE_MLA_ERR_CUDA;
  p.valid_count = counts;
  smla::valid_count_kernel<<<p.ctas, smla::kProducerWarps * 32, 0, cs>>>(p);
  return cudaGetLastError() == cudaSuccess ? SPARSE_MLA_OK : SPARSE_MLA_ERR_CUDA;
}

sparse_mla_status_t check_count_args(const int32_t* indices, long long n_tok, int topk, const int32_t* counts) {
  if (n_tok < 0 || topk < 1 || n_tok > INT_MAX / 2) return SPARSE_MLA_ERR_INVALID_ARG;
  if (n_tok > 0 && (!indices || !counts || !aligned(indices, 4) || !aligned(counts, 4)))
    return SPARSE_MLA_ERR_INVALID_ARG;
  return SPARSE_MLA_OK;
}

}  // namespace

extern "C" {

sparse_mla_status_t sparse_mla_debug_valid_count(const int32_t* indices, int s_q, int s_kv, int topk,
                                                 int32_t* counts, void* stream) {
  sparse_mla_status_t st = check_count_args(indices, s_q, topk, counts);
  if (st != SPARSE_MLA_OK) return st;
  if (s_kv < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_setup(&sms)) != SPARSE_MLA_OK) return st;
  if (s_q == 0) return SPARSE_MLA_OK;
  FwdParams p = base_params(nullptr, indices, 1.f, nullptr, nullptr, s_q, 1, topk);
  p.mode = smla::kDense;
  p.n_rows = s_kv;
  p.s_kv = s_kv;
  p.sched = smla::kWholeUnits;
  p.ctas = prefill_ctas(s_q, 1, sms);
  return launch_valid_count(p, counts, static_cast<cudaStream_t>(stream));
}

sparse_mla_status_t sparse_mla_debug_valid_count_varlen(const int32_t* indices, const int32_t* cu_seqlens_q,
                                                        const int32_t* cu_seqlens_kv, int batch, int total_q,
                                                        int total_kv, int topk, int32_t* counts, void* stream) {
  sparse_mla_status_t st = check_count_args(indices, total_q, topk, counts);
  if (st != SPARSE_MLA_OK) return st;
  if (total_kv < 0 || batch < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  if (total_q > 0 && (batch < 1 || !cu_seqlens_q || !cu_seqlens_kv || !aligned(cu_seqlens_q, 4) ||
                      !aligned(cu_seqlens_kv, 4)))
    return SPARSE_MLA_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_setup(&sms)) != SPARSE_MLA_OK) return st;
  if (total_q == 0) return SPARSE_MLA_OK;
  FwdParams p = base_params(nullptr, indices, 1.f, nullptr, nullptr, total_q, 1, topk);
  p.mode = smla::kVarlen;
  p.n_rows = total_kv;
  p.batch = batch;
  p.cu_q = cu_seqlens_q;
  p.cu_kv = cu_seqlens_kv;
  p.sched = smla::kWholeUnits;
  p.ctas = prefill_ctas(total_q, 1, sms);
  return launch_valid_count(p, counts, static_cast<cudaStream_t>(stream));
}

sparse_mla_status_t sparse_mla_debug_valid_count_paged(const int32_t* indices, const int32_t* block_table,
                                                       const int32_t* cache_seqlens, int batch, int s_next, int topk,
                                                       int page_size, int max_blocks, int num_blocks,
                                                       int32_t* counts, void* stream) {
  if (batch < 0 || s_next < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  const long long n_tok = static_cast<long long>(batch) * s_next;
  sparse_mla_status_t st = check_count_args(indices, n_tok, topk, counts);
  if (st != SPARSE_MLA_OK) return st;
  if (page_size < 1 || max_blocks < 0 || num_blocks < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  if (static_cast<long long>(num_blocks) * page_size > INT_MAX) return SPARSE_MLA_ERR_INVALID_ARG;
  if (n_tok > 0 && (!block_table || !cache_seqlens || !aligned(block_table, 4) || !aligned(cache_seqlens, 4)))
    return SPARSE_MLA_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_setup(&sms)) != SPARSE_MLA_OK) return st;
  if (n_tok == 0) return SPARSE_MLA_OK;
  if (n_tok * blocks_per_list(topk) > (1LL << 62) / (sms > 0 ? sms : 1)) return SPARSE_MLA_ERR_INVALID_ARG;
  FwdParams p = base_params(nullptr, indices, 1.f, nullptr, nullptr, static_cast<int>(n_tok), 1, topk);
  p.mode = smla::kPaged;
  p.n_rows = num_blocks * page_size;
  p.batch = batch;
  p.s_next = s_next;
  p.page_size = page_size;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  p.block_table = block_table;
  p.seqlens = cache_seqlens;
  // The block ranges of a decode launch (one head group), so the walk cuts
  // the lists where the forward does.
  p.sched = smla::kBlockRanges;
  p.ctas = decode_ctas(n_tok, 1, topk, sms);
  return launch_valid_count(p, counts, static_cast<cudaStream_t>(stream));
}

const char* sparse_mla_status_string(sparse_mla_status_t s) {
  switch (s) {
    case SPARSE_MLA_OK: return "SPARSE_MLA_OK";
    case SPARSE_MLA_ERR_INVALID_ARG: return "SPARSE_MLA_ERR_INVALID_ARG";
    case SPARSE_MLA_ERR_UNSUPPORTED_SHAPE: return "SPARSE_MLA_ERR_UNSUPPORTED_SHAPE";
    case SPARSE_MLA_ERR_UNSUPPORTED_ARCH: return "SPARSE_MLA_ERR_UNSUPPORTED_ARCH";
    case SPARSE_MLA_ERR_CUDA: return "SPARSE_MLA_ERR_CUDA";
    case SPARSE_MLA_ERR_DEVICE_TIMEOUT: return "SPARSE_MLA_ERR_DEVICE_TIMEOUT";
    case SPARSE_MLA_ERR_WORKSPACE_TOO_SMALL: return "SPARSE_MLA_ERR_WORKSPACE_TOO_SMALL";
  }
  return "SPARSE_MLA_UNKNOWN_STATUS";
}

sparse_mla_status_t sparse_mla_get_device_error(int* code) {
  if (!code) return SPARSE_MLA_ERR_INVALID_ARG;
  int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return SPARSE_MLA_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&v, smla::g_device_error, sizeof(int)) != cudaSuccess) return SPARSE_MLA_ERR_CUDA;
  *code = v;
  return SPARSE_MLA_OK;
}

sparse_mla_status_t sparse_mla_clear_device_error(void) {
  const int zero = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return SPARSE_MLA_ERR_CUDA;
  if (cudaMemcpyToSymbol(smla::g_device_error, &zero, sizeof(int)) != cudaSuccess) return SPARSE_MLA_ERR_CUDA;
  return SPARSE_MLA_OK;
}

void sparse_mla_set_wait_timeout_ns(unsigned long long ns) { g_timeout_ns.store(ns ? ns : kDefaultTimeoutNs); }

}  // extern "C"

// ------------------------------------------------------------------ DSA indexer

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

sparse_mla_status_t get_encode(EncodeTiledFn* fn) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || f == nullptr)
      return SPARSE_MLA_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(f);
  }
  *fn = g_encode;
  return SPARSE_MLA_OK;
}

// A 2-D bf16 tensor [rows, 128] read in boxes of 64 columns x box_rows rows,
// 128B-swizzled (the K-major layout the MMA descriptors expect); boxes past
// the last row read zeros.
sparse_mla_status_t encode_rows128(EncodeTiledFn enc, CUtensorMap* map, const void* base, long long rows,
                                   int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(smla::kIdxD), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(smla::kIdxD) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SPARSE_MLA_OK : SPARSE_MLA_ERR_INVALID_ARG;
}

bool idx_heads_ok(int h_idx) { return h_idx == 16 || h_idx == 32 || h_idx == 64; }

// Shape and pointer checks shared by the indexer entry points.
sparse_mla_status_t check_indexer(const void* q_idx, const void* k_idx, const float* weights,
                                  const int32_t* cu_q, const int32_t* cu_kv, int batch, int total_q, int total_kv,
                                  int h_idx, int d_idx) {
  if (total_q < 0 || total_kv < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  if (d_idx != smla::kIdxD || !idx_heads_ok(h_idx)) return SPARSE_MLA_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(total_q) * h_idx + smla::kIdxN > INT_MAX ||
      static_cast<long long>(total_kv) + smla::kIdxTile * smla::kIdxChunkTiles > INT_MAX)
    return SPARSE_MLA_ERR_INVALID_ARG;
  if ((cu_q == nullptr) != (cu_kv == nullptr)) return SPARSE_MLA_ERR_INVALID_ARG;
  if (cu_q != nullptr) {
    if (batch < 1 || !aligned(cu_q, 4) || !aligned(cu_kv, 4)) return SPARSE_MLA_ERR_INVALID_ARG;
    if (batch > smla::kIdxMaxBatch) return SPARSE_MLA_ERR_UNSUPPORTED_SHAPE;
  }
  if (total_q > 0 && total_kv > 0) {
    if (!q_idx || !k_idx || !weights) return SPARSE_MLA_ERR_INVALID_ARG;
    if (!aligned(q_idx, 16) || !aligned(k_idx, 16) || !aligned(weights, 16)) return SPARSE_MLA_ERR_INVALID_ARG;
  }
  return SPARSE_MLA_OK;
}

// How a launch's query rows map to key sequences: one dense sequence (all
// null), packed sequences (cu_q / cu_kv) or a paged decode cache
// (block_table / seqlens, s_next rows per request).
struct IdxSeqs {
  const int32_t* cu_q = nullptr;
  const int32_t* cu_kv = nullptr;
  const int32_t* block_table = nullptr;
  const int32_t* seqlens = nullptr;
  int batch = 1, s_next = 0, max_blocks = 0, num_blocks = 0;
};

sparse_mla_status_t launch_scores(const void* q_idx, const void* k_idx, const float* weights, const IdxSeqs& sq,
                                  int total_q, int total_kv, int h_idx, int row0, int n_rows, int skip_len,
                                  float* scores, long long row_stride, int sms, cudaStream_t cs) {
  if (n_rows <= 0 || total_kv <= 0) return SPARSE_MLA_OK;
  EncodeTiledFn enc = nullptr;
  sparse_mla_status_t st = get_encode(&enc);
  if (st != SPARSE_MLA_OK) return st;
  smla::IdxParams p;
  std::memset(&p, 0, sizeof(p));
  if ((st = encode_rows128(enc, &p.map_q, q_idx, static_cast<long long>(total_q) * h_idx, smla::kIdxN)) !=
      SPARSE_MLA_OK)
    return st;
  const bool paged = sq.block_table != nullptr;
  if ((st = encode_rows128(enc, &p.map_k, k_idx, total_kv, paged ? smla::kIdxPage : smla::kIdxTile)) != SPARSE_MLA_OK)
    return st;
  p.weights = weights;
  p.cu_q = sq.cu_q;
  p.cu_kv = sq.cu_kv;
  p.block_table = sq.block_table;
  p.seqlens = sq.seqlens;
  p.s_next = sq.s_next;
  p.max_blocks = sq.max_blocks;
  p.num_blocks = sq.num_blocks;
  p.scores = scores;
  p.row_stride = row_stride;
  p.total_q = total_q;
  p.total_kv = total_kv;
  p.batch = (sq.cu_q || paged) ? sq.batch : 1;
  p.h_idx = h_idx;
  p.row0 = row0;
  p.n_rows = n_rows;
  p.skip_len = skip_len;
  const int G = smla::kIdxN / h_idx;
  p.groups = (n_rows + G - 1) / G;
  const long long longest = row_stride < total_kv || paged ? row_stride : total_kv;
  // Tiles per item: about four items per SM over the (at most) groups x
  // tiles of the launch, between 4 and 32 tiles, a power of two.
  const long long tiles = static_cast<long long>(p.groups) * ((longest + smla::kIdxTile - 1) / smla::kIdxTile);
  int ct = smla::kIdxChunkTiles;
  while (ct > 4 && tiles / ct < 4LL * sms) ct >>= 1;
  p.chunk_tiles = ct;
  const long long span = static_cast<long long>(smla::kIdxTile) * ct;
  p.kv_chunks = static_cast<int>((longest + span - 1) / span);
  if (p.kv_chunks < 1) p.kv_chunks = 1;
  unsigned long long t = g_timeout_ns.load();
  p.timeout_ns = t ? t : kDefaultTimeoutNs;
  const long long items = static_cast<long long>(p.groups) * p.kv_chunks;
  const int ctas = static_cast<int>(items < sms ? items : sms);
  if (h_idx == 16)
    smla::dsa_scores_kernel<16><<<ctas, smla::kIdxThreads, smla::idx_smem_bytes(), cs>>>(p);
  else if (h_idx == 32)
    smla::dsa_scores_kernel<32><<<ctas, smla::kIdxThreads, smla::idx_smem_bytes(), cs>>>(p);
  else
    smla::dsa_scores_kernel<64><<<ctas, smla::kIdxThreads, smla::idx_smem_bytes(), cs>>>(p);
  return cudaGetLastError() == cudaSuccess ? SPARSE_MLA_OK : SPARSE_MLA_ERR_CUDA;
}

sparse_mla_status_t launch_topk(const float* scores, long long row_stride, const IdxSeqs& sq, int total_q,
                                int total_kv, int row0, int n_rows, int topk, int32_t* indices, cudaStream_t cs) {
  if (n_rows <= 0) return SPARSE_MLA_OK;
  smla::TopkParams p;
  std::memset(&p, 0, sizeof(p));
  const bool paged = sq.block_table != nullptr;
  p.scores = scores;
  p.indices = indices;
  p.cu_q = paged ? nullptr : sq.cu_q;
  p.cu_kv = paged ? nullptr : sq.cu_kv;
  p.seqlens = paged ? sq.seqlens : nullptr;
  p.block_table = paged ? sq.block_table : nullptr;
  p.max_blocks = sq.max_blocks;
  p.num_blocks = sq.num_blocks;
  p.s_next = sq.s_next;
  p.row_stride = row_stride;
  p.total_q = total_q;
  p.total_kv = total_kv;
  p.batch = (sq.cu_q || paged) ? sq.batch : 1;
  p.row0 = row0;
  p.n_rows = n_rows;
  p.topk = topk;
  const long long longest = row_stride < total_kv || paged ? row_stride : total_kv;
  p.stage_cap = static_cast<int>(longest < kTopkStageCap ? (longest + 3) / 4 * 4 : kTopkStageCap);
  const int smem = smla::kTopkBins * 4 + p.stage_cap * 4;
  // Rows beyond 8192 positions (decode over long contexts) take CTAs of 1024
  // threads: few rows, each with more work.
  if (longest > 8192)
    smla::dsa_topk_kernel<1024><<<n_rows, 1024, smem, cs>>>(p);
  else
    smla::dsa_topk_kernel<256><<<n_rows, 256, smem, cs>>>(p);
  return cudaGetLastError() == cudaSuccess ? SPARSE_MLA_OK : SPARSE_MLA_ERR_CUDA;
}

long long idx_row_stride(int max_seqlen_kv) { return (static_cast<long long>(max_seqlen_kv) + 3) / 4 * 4; }

IdxSeqs paged_seqs(const int32_t* block_table, const int32_t* seqlens, int batch, int s_next, int max_blocks,
                   int num_blocks) {
  IdxSeqs sq;
  sq.block_table = block_table;
  sq.seqlens = seqlens;
  sq.batch = batch;
  sq.s_next = s_next;
  sq.max_blocks = max_blocks;
  sq.num_blocks = num_blocks;
  return sq;
}

sparse_mla_status_t check_paged_indexer(const void* q_idx, const void* k_cache, const float* weights,
                                        const int32_t* block_table, const int32_t* seqlens, int batch, int s_next,
                                        int h_idx, int d_idx, int page_size, int max_blocks, int num_blocks) {
  if (batch < 0 || s_next < 1 || max_blocks < 0 || num_blocks < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  if (d_idx != smla::kIdxD || !idx_heads_ok(h_idx) || page_size != smla::kIdxPage)
    return SPARSE_MLA_ERR_UNSUPPORTED_SHAPE;
  if (batch > smla::kIdxMaxBatch) return SPARSE_MLA_ERR_UNSUPPORTED_SHAPE;
  const long long total_q = static_cast<long long>(batch) * s_next;
  if (total_q * h_idx + smla::kIdxN > INT_MAX ||
      static_cast<long long>(num_blocks) * smla::kIdxPage + smla::kIdxTile * smla::kIdxChunkTiles > INT_MAX)
    return SPARSE_MLA_ERR_INVALID_ARG;
  if (batch > 0) {
    if (!q_idx || !weights || !block_table || !seqlens) return SPARSE_MLA_ERR_INVALID_ARG;
    if (!aligned(q_idx, 16) || !aligned(weights, 16) || !aligned(block_table, 4) || !aligned(seqlens, 4))
      return SPARSE_MLA_ERR_INVALID_ARG;
    if (num_blocks > 0 && (!k_cache || !aligned(k_cache, 16))) return SPARSE_MLA_ERR_INVALID_ARG;
  }
  return SPARSE_MLA_OK;
}

// Scores and lists of every query row, in chunks of rows whose logits fit the
// workspace (the logits budget); rows before first_long are known to be short.
sparse_mla_status_t indexer_topk_chunks(const void* q_idx, const void* k_idx, const float* weights, const IdxSeqs& sq,
                                        int total_q, int total_kv, int max_seqlen_kv, int h_idx, int topk,
                                        long long first_long, int32_t* indices, void* workspace,
                                        size_t workspace_bytes, cudaStream_t cs) {
  if (static_cast<long long>(total_q) * topk > (1LL << 62)) return SPARSE_MLA_ERR_INVALID_ARG;
  if (total_q > 0 && (!indices || !aligned(indices, 4))) return SPARSE_MLA_ERR_INVALID_ARG;
  int sms = 0;
  sparse_mla_status_t st = device_setup(&sms);
  if (st != SPARSE_MLA_OK) return st;
  if (total_q == 0) return SPARSE_MLA_OK;
  if (max_seqlen_kv <= topk)   // every row is short: identity lists, no scores
    return launch_topk(nullptr, 1, sq, total_q, total_kv, 0, total_q, topk, indices, cs);
  const long long stride = idx_row_stride(max_seqlen_kv);
  if (!workspace || !aligned(workspace, 16)) return SPARSE_MLA_ERR_WORKSPACE_TOO_SMALL;
  long long rows = static_cast<long long>(workspace_bytes / (static_cast<size_t>(stride) * sizeof(float)));
  if (rows < 1) return SPARSE_MLA_ERR_WORKSPACE_TOO_SMALL;
  if (rows > total_q) rows = total_q;
  float* ws = static_cast<float*>(workspace);
  for (long long r0 = 0; r0 < total_q; r0 += rows) {
    const int n = static_cast<int>(total_q - r0 < rows ? total_q - r0 : rows);
    if (r0 + n > first_long) {
      const long long s0 = r0 > first_long ? r0 : first_long;   // scored rows of this chunk start here
      if ((st = launch_scores(q_idx, k_idx, weights, sq, total_q, total_kv, h_idx, static_cast<int>(s0),
                              static_cast<int>(r0 + n - s0), topk, ws + (s0 - r0) * stride, stride, sms, cs)) !=
          SPARSE_MLA_OK)
        return st;
    }
    if ((st = launch_topk(ws, stride, sq, total_q, total_kv, static_cast<int>(r0), n, topk, indices, cs)) !=
        SPARSE_MLA_OK)
      return st;
  }
  return SPARSE_MLA_OK;
}

}  // namespace

extern "C" {

sparse_mla_status_t dsa_indexer_scores(const void* q_idx, const void* k_idx, const float* weights,
                                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch,
                                       int total_q, int total_kv, int h_idx, int d_idx, int row0, int n_rows,
                                       int skip_len, float* scores, long long row_stride, void* stream) {
  sparse_mla_status_t st = check_indexer(q_idx, k_idx, weights, cu_seqlens_q, cu_seqlens_kv, batch, total_q,
                                         total_kv, h_idx, d_idx);
  if (st != SPARSE_MLA_OK) return st;
  if (row0 < 0 || n_rows < 0 || static_cast<long long>(row0) + n_rows > total_q || skip_len < 0 || row_stride < 1)
    return SPARSE_MLA_ERR_INVALID_ARG;
  if (n_rows > 0 && total_kv > 0 && (!scores || !aligned(scores, 4))) return SPARSE_MLA_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_setup(&sms)) != SPARSE_MLA_OK) return st;
  IdxSeqs sq;
  sq.cu_q = cu_seqlens_q;
  sq.cu_kv = cu_seqlens_kv;
  sq.batch = batch;
  return launch_scores(q_idx, k_idx, weights, sq, total_q, total_kv, h_idx, row0, n_rows, skip_len, scores,
                       row_stride, sms, static_cast<cudaStream_t>(stream));
}

sparse_mla_status_t dsa_topk(const float* scores, long long row_stride, const int32_t* cu_seqlens_q,
                             const int32_t* cu_seqlens_kv, int batch, int total_q, int total_kv, int row0,
                             int n_rows, int topk, int32_t* indices, void* stream) {
  if (total_q < 0 || total_kv < 0 || topk < 1 || row0 < 0 || n_rows < 0 ||
      static_cast<long long>(row0) + n_rows > total_q || row_stride < 1)
    return SPARSE_MLA_ERR_INVALID_ARG;
  if ((cu_seqlens_q == nullptr) != (cu_seqlens_kv == nullptr)) return SPARSE_MLA_ERR_INVALID_ARG;
  if (cu_seqlens_q != nullptr && (batch < 1 || !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_kv, 4)))
    return SPARSE_MLA_ERR_INVALID_ARG;
  if (static_cast<long long>(total_q) * topk > (1LL << 62)) return SPARSE_MLA_ERR_INVALID_ARG;
  if (n_rows > 0 && (!indices || !aligned(indices, 4))) return SPARSE_MLA_ERR_INVALID_ARG;
  if (n_rows > 0 && total_kv > topk && (!scores || !aligned(scores, 4))) return SPARSE_MLA_ERR_INVALID_ARG;
  int sms = 0;
  sparse_mla_status_t st = device_setup(&sms);
  if (st != SPARSE_MLA_OK) return st;
  IdxSeqs sq;
  sq.cu_q = cu_seqlens_q;
  sq.cu_kv = cu_seqlens_kv;
  sq.batch = batch;
  return launch_topk(scores, row_stride, sq, total_q, total_kv, row0, n_rows, topk, indices,
                     static_cast<cudaStream_t>(stream));
}

size_t dsa_indexer_workspace_size(int total_q, int max_seqlen_kv, int topk) {
  if (total_q < 1 || max_seqlen_kv < 1 || topk < 1 || max_seqlen_kv <= topk) return 0;
  return static_cast<size_t>(total_q) * static_cast<size_t>(idx_row_stride(max_seqlen_kv)) * sizeof(float);
}

sparse_mla_status_t dsa_indexer_topk(const void* q_idx, const void* k_idx, const float* weights,
                                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int batch,
                                     int total_q, int total_kv, int max_seqlen_kv, int h_idx, int d_idx, int topk,
                                     int32_t* indices, void* workspace, size_t workspace_bytes, void* stream) {
  sparse_mla_status_t st = check_indexer(q_idx, k_idx, weights, cu_seqlens_q, cu_seqlens_kv, batch, total_q,
                                         total_kv, h_idx, d_idx);
  if (st != SPARSE_MLA_OK) return st;
  if (topk < 1 || max_seqlen_kv < 0 || max_seqlen_kv > total_kv) return SPARSE_MLA_ERR_INVALID_ARG;
  if (cu_seqlens_q == nullptr && max_seqlen_kv != total_kv) return SPARSE_MLA_ERR_INVALID_ARG;
  IdxSeqs sq;
  sq.cu_q = cu_seqlens_q;
  sq.cu_kv = cu_seqlens_kv;
  sq.batch = batch;
  // One dense sequence: rows before first_long see at most topk positions.
  long long first_long = 0;
  if (cu_seqlens_q == nullptr) {
    first_long = static_cast<long long>(topk) - (total_kv - total_q);
    if (first_long < 0) first_long = 0;
    if (first_long > total_q) first_long = total_q;
  }
  return indexer_topk_chunks(q_idx, k_idx, weights, sq, total_q, total_kv, max_seqlen_kv, h_idx, topk, first_long,
                             indices, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

sparse_mla_status_t dsa_indexer_scores_paged(const void* q_idx, const void* k_cache, const float* weights,
                                             const int32_t* block_table, const int32_t* cache_seqlens, int batch,
                                             int s_next, int h_idx, int d_idx, int page_size, int max_blocks,
                                             int num_blocks, int row0, int n_rows, int skip_len, float* scores,
                                             long long row_stride, void* stream) {
  sparse_mla_status_t st = check_paged_indexer(q_idx, k_cache, weights, block_table, cache_seqlens, batch, s_next,
                                               h_idx, d_idx, page_size, max_blocks, num_blocks);
  if (st != SPARSE_MLA_OK) return st;
  const long long total_q = static_cast<long long>(batch) * s_next;
  if (row0 < 0 || n_rows < 0 || row0 + static_cast<long long>(n_rows) > total_q || skip_len < 0 || row_stride < 1)
    return SPARSE_MLA_ERR_INVALID_ARG;
  if (n_rows > 0 && (!scores || !aligned(scores, 4))) return SPARSE_MLA_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_setup(&sms)) != SPARSE_MLA_OK) return st;
  IdxSeqs sq = paged_seqs(block_table, cache_seqlens, batch, s_next, max_blocks, num_blocks);
  return launch_scores(q_idx, k_cache, weights, sq, static_cast<int>(total_q), num_blocks * smla::kIdxPage, h_idx,
                       row0, n_rows, skip_len, scores, row_stride, sms, static_cast<cudaStream_t>(stream));
}

sparse_mla_status_t dsa_indexer_topk_paged(const void* q_idx, const void* k_cache, const float* weights,
                                           const int32_t* block_table, const int32_t* cache_seqlens, int batch,
                                           int s_next, int h_idx, int d_idx, int page_size, int max_blocks,
                                           int num_blocks, int max_seqlen_kv, int topk, int32_t* indices,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  sparse_mla_status_t st = check_paged_indexer(q_idx, k_cache, weights, block_table, cache_seqlens, batch, s_next,
                                               h_idx, d_idx, page_size, max_blocks, num_blocks);
  if (st != SPARSE_MLA_OK) return st;
  if (topk < 1 || max_seqlen_kv < 0) return SPARSE_MLA_ERR_INVALID_ARG;
  const long long total_q = static_cast<long long>(batch) * s_next;
  IdxSeqs sq = paged_seqs(block_table, cache_seqlens, batch, s_next, max_blocks, num_blocks);
  return indexer_topk_chunks(q_idx, k_cache, weights, sq, static_cast<int>(total_q), num_blocks * smla::kIdxPage,
                             max_seqlen_kv, h_idx, topk, 0, indices, workspace, workspace_bytes,
                             static_cast<cudaStream_t>(stream));
}

}  // extern "C"

// attn_append_kv: the step before attention on every mode — the new tokens'
// K and V rows go into their pages of the paged caches.
//
// Request b's new token t sits at position i = seq_lens[b] - n_b + t (the
// bottom-right reading the attention kernels use), i.e. page
// page_table[b][i / P], offset i % P.  BF16 caches take the rows bit for bit;
// FP8 caches take E4M3 codes of value / scale, the division in fp32 and the
// conversion round-to-nearest-even with saturation to +-448, which is how an
// FP8 E4M3 KV cache with a per-tensor scale stores its entries (model card
// MiMo-V2.6-Flash-RL-FP8KV-W4A8-2x-RTX-PRO-6000, "What the kernels do").
//
// One thread per 16-byte chunk of a source row (8 bf16 values): a row of K is
// 24 chunks, a row of V 16; the thread finds its request by binary search in
// qo_indptr.  The kernel streams its bytes once (HBM-bound for large appends,
// launch-bound for decode-sized ones).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_paged.h"
#include "plan.hpp"

namespace akp {
namespace {

constexpr int kVChunks = kDv / 8;    // 16-byte bf16 chunks of a V row: 16

struct AppendArgs {
  const uint16_t *k_new, *v_new;
  void *k_cache, *v_cache;
  const int32_t *page_table, *seq_lens, *qo_indptr;
  int32_t *err;
  int64_t units;            // total_q * hkv * (k_chunks + 16)
  int32_t batch, hkv, page_size, pt_stride, num_pages;
  int32_t dqk, k_chunks;    // query/key head dim, 16-byte chunks of a K row (dqk / 8)
  int32_t qo_in_smem;       // nonzero: the launch gives (batch + 1) * 4 bytes of shared memory
  float k_scale, v_scale;
};

// Two fp32 values -> two E4M3 codes (RNE, saturating), low byte = lo.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

template <bool FP8>
__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a) {
  // the kernels that follow in a serving step (device planner, attention) may
  // be scheduled now; they wait for this grid before reading the caches
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  // qo_indptr in shared memory when it fits (the launch passes the size): the
  // request of a token is then found without a chain of dependent global loads
  extern __shared__ int32_t s_qo[];
  const bool qo_smem = a.qo_in_smem != 0;
  if (qo_smem) {
    for (int i = threadIdx.x; i <= a.batch; i += blockDim.x) s_qo[i] = __ldg(a.qo_indptr + i);
    __syncthreads();
  }
  auto qo_at = [&](int i) { return qo_smem ? s_qo[i] : __ldg(a.qo_indptr + i); };
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < a.units;
       u += (int64_t)gridDim.x * blockDim.x) {
    const int chunks = a.k_chunks + kVChunks;
    const int chunk = (int)(u % chunks);
    const int64_t pair = u / chunks;
    const int g = (int)(pair % a.hkv);
    const int tok = (int)(pair / a.hkv);
    // the source chunk depends on nothing that follows: its load goes out first
    const bool is_k = chunk < a.k_chunks;
    const int c = is_k ? chunk : chunk - a.k_chunks;
    const int D = is_k ? a.dqk : kDv;
    const uint4 src = __ldg(reinterpret_cast<const uint4 *>((is_k ? a.k_new : a.v_new) +
                                                            ((int64_t)tok * a.hkv + g) * D) + c);
    // request of this token: last b with qo_indptr[b] <= tok
    int lo = 0, hi = a.batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (qo_at(mid) <= tok) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int q0 = qo_at(b), n = qo_at(b + 1) - q0;
    const int64_t i = (int64_t)__ldg(a.seq_lens + b) - n + (tok - q0);
    if (i < 0 || i / a.page_size >= a.pt_stride) {   // a length outside the table row
      atomicOr(a.err, 4);
      continue;
    }
    const int32_t page = __ldg(a.page_table + (int64_t)b * a.pt_stride + i / a.page_size);
    if (page < 0 || page >= a.num_pages) {
      atomicOr(a.err, 1);
      continue;
    }
    const int64_t slot = (int64_t)page * a.page_size + i % a.page_size;
    const int64_t row = (slot * a.hkv + g) * D;
    if (!FP8) {
      reinterpret_cast<uint4 *>(static_cast<uint16_t *>(is_k ? a.k_cache : a.v_cache) + row)[c] =
          src;
    } else {
      const float s = is_k ? a.k_scale : a.v_scale;
      const uint32_t w[4] = {src.x, src.y, src.z, src.w};
      uint32_t out[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float f[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          f[2 * e] = __fdiv_rn(__uint_as_float(w[2 * h + e] << 16), s);
          f[2 * e + 1] = __fdiv_rn(__uint_as_float(w[2 * h + e] & 0xFFFF0000u), s);
        }
        out[h] = (uint32_t)e4m3x2(f[0], f[1]) | ((uint32_t)e4m3x2(f[2], f[3]) << 16);
      }
      reinterpret_cast<uint2 *>(static_cast<uint8_t *>(is_k ? a.k_cache : a.v_cache) + row)[c] =
          make_uint2(out[0], out[1]);
    }
  }
}

}  // namespace
}  // namespace akp

extern "C" attn_status_t attn_append_kv(attn_plan_t plan, const void *k_new, const void *v_new,
                                        void *k_cache, void *v_cache, const int32_t *page_table,
                                        const int32_t *seq_lens, const int32_t *qo_indptr,
                                        float k_scale, float v_scale, void *stream) {
  if (!plan || plan->device < 0) return ATTN_ERR_INVALID_ARG;
  const akp::HostPlan &hp = plan->host;
  const attn_problem_t &pr = hp.prob;
  const int64_t total_q = hp.qo_indptr.back();
  if (total_q == 0) return ATTN_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !page_table || !seq_lens || !qo_indptr)
    return ATTN_ERR_INVALID_ARG;
  const bool fp8 = pr.kv_dtype == ATTN_KV_FP8_E4M3;
  if (fp8 && !(k_scale > 0.f && v_scale > 0.f && k_scale < INFINITY && v_scale < INFINITY))
    return ATTN_ERR_INVALID_ARG;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (prev != plan->device && cudaSetDevice(plan->device) != cudaSuccess) return ATTN_ERR_CUDA;
  akp::AppendArgs a{};
  a.k_new = static_cast<const uint16_t *>(k_new);
  a.v_new = static_cast<const uint16_t *>(v_new);
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.qo_indptr = qo_indptr;
  a.err = plan->dev.err;
  a.dqk = pr.head_dim_qk;
  a.k_chunks = pr.head_dim_qk / 8;
  a.units = total_q * pr.num_kv_heads * (a.k_chunks + akp::kVChunks);
  a.batch = pr.batch;
  a.hkv = pr.num_kv_heads;
  a.page_size = pr.page_size;
  a.pt_stride = pr.page_table_stride;
  a.num_pages = pr.num_pages;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  const int64_t want = (a.units + 255) / 256;
  const unsigned grid = (unsigned)(want < 152 * 16 ? want : 152 * 16);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t qo_bytes = (size_t)(pr.batch + 1) * sizeof(int32_t);
  a.qo_in_smem = qo_bytes <= 16 * 1024;
  const size_t smem = a.qo_in_smem ? qo_bytes : 0;
  if (fp8)
    akp::append_kernel<true><<<grid, 256, smem, st>>>(a);
  else
    akp::append_kernel<false><<<grid, 256, smem, st>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (prev != plan->device) cudaSetDevice(prev);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Single-token Gated DeltaNet step with the state updated in place (sm_103a).
//
// For each (sequence, value head), one token:
//   S <- alpha S;   u = beta (v - S k);   S <- S + u k^T;   o = S q / sqrt(dk)
// which is the recurrence S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T,
// o_t = S_t q_t / sqrt(dk) applied to one token after a prefill has produced the
// state ("chunked Gated DeltaNet prefill" of the "Open-Jev-27B-v1.1 native text
// worker" page; the pages' workers score prompts and generate nothing, so this
// is the adjacent decode form of the same operation).
//
// The step reads and writes the whole fp32 state once and does two dot products
// per state row, so it is bound by HBM bandwidth: a warp takes four state rows at a
// time, each lane holding dk / 32 consecutive elements of a row (16-byte loads and
// stores for dk = 128), the two row reductions by warp shuffles.  Tensor cores would
// not help a matrix-vector step.
#include "gdn_common.cuh"

namespace gdn {

namespace {
constexpr int kDecodeWarps = 8;
constexpr int kRowsPerBatch = 4;  // rows a warp has in flight together
}  // namespace

// One CTA per (sequence, value head): warp w walks state rows w * DV / 8 .. (w + 1) * DV / 8 - 1
// in batches of four, the next batch's loads issued before the current batch is computed.
template <int DK>
__global__ void __launch_bounds__(32 * kDecodeWarps)
gdn_decode_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                  const __nv_bfloat16* __restrict__ v, const float* __restrict__ g,
                  const float* __restrict__ beta, float* __restrict__ state, __nv_bfloat16* __restrict__ out,
                  int Hk, int Hv, int DV) {
  constexpr int E = DK / 32;  // state elements per lane
  constexpr int R = kRowsPerBatch;
  const int bh = blockIdx.x;  // sequence * Hv + value head
  const int b = bh / Hv, h = bh - b * Hv;
  const int hk = h / (Hv / Hk);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float alpha = expf(g[bh]);
  const float bt = beta[bh];
  const float scale = rsqrtf((float)DK);

  float kv[E], qv[E];
  const __nv_bfloat16* kr = k + ((size_t)b * Hk + hk) * DK + lane * E;
  const __nv_bfloat16* qr = q + ((size_t)b * Hk + hk) * DK + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    kv[e] = __bfloat162float(kr[e]);
    qv[e] = __bfloat162float(qr[e]);
  }

  const int rows_per_warp = DV / kDecodeWarps;  // 4, 8 or 16
  const int nbatch = rows_per_warp / R;
  const int row_base = warp * rows_per_warp;
  float* srow0 = state + ((size_t)bh * DV + row_base) * DK + lane * E;
  auto load = [&](float (&x)[R][E], int j) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float* p = srow0 + (size_t)(j * R + r) * DK;
      if constexpr (E == 4) {
        const float4 t = *reinterpret_cast<const float4*>(p);
        x[r][0] = t.x; x[r][1] = t.y; x[r][2] = t.z; x[r][3] = t.w;
      } else if constexpr (E == 2) {
        const float2 t = *reinterpret_cast<const float2*>(p);
        x[r][0] = t.x; x[r][1] = t.y;
      } else {
        x[r][0] = p[0];
      }
    }
  };
  float sv[R][E], nx[R][E];
  load(sv, 0);
  for (int j = 0; j < nbatch; ++j) {
    if (j + 1 < nbatch) load(nx, j + 1);
    // decay, then the prediction S k of every row
    float sk[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        sv[r][e] *= alpha;
        acc = fmaf(sv[r][e], kv[e], acc);
      }
      sk[r] = acc;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int r = 0; r < R; ++r) sk[r] += __shfl_xor_sync(0xffffffffu, sk[r], o);
    // rank-one write, then the output S q
    const int row0 = row_base + j * R;
    float sq[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float vr = __bfloat162float(v[(size_t)bh * DV + row0 + r]);
      const float u = bt * (vr - sk[r]);
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        sv[r][e] = fmaf(u, kv[e], sv[r][e]);
        acc = fmaf(sv[r][e], qv[e], acc);
      }
      sq[r] = acc;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int r = 0; r < R; ++r) sq[r] += __shfl_xor_sync(0xffffffffu, sq[r], o);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float* p = srow0 + (size_t)(j * R + r) * DK;
      if constexpr (E == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(sv[r][0], sv[r][1], sv[r][2], sv[r][3]);
      } else if constexpr (E == 2) {
        *reinterpret_cast<float2*>(p) = make_float2(sv[r][0], sv[r][1]);
      } else {
        p[0] = sv[r][0];
      }
      if (lane == 0) out[(size_t)bh * DV + row0 + r] = __float2bfloat16_rn(sq[r] * scale);
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int e = 0; e < E; ++e) sv[r][e] = nx[r][e];
  }
}

template <int DK>
cudaError_t launch_decode(const void* q, const void* k, const void* v, const float* g, const float* beta,
                          float* state, void* out, int B, int Hk, int Hv, int DV, cudaStream_t st) {
  if (DV % (kDecodeWarps * kRowsPerBatch) != 0) return cudaErrorInvalidValue;
  gdn_decode_kernel<DK><<<(unsigned)B * Hv, 32 * kDecodeWarps, 0, st>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), g, beta, state, static_cast<__nv_bfloat16*>(out), Hk, Hv, DV);
  return cudaGetLastError();
}

template cudaError_t launch_decode<32>(const void*, const void*, const void*, const float*, const float*, float*,
                                       void*, int, int, int, int, cudaStream_t);
template cudaError_t launch_decode<64>(const void*, const void*, const void*, const float*, const float*, float*,
                                       void*, int, int, int, int, cudaStream_t);
template cudaError_t launch_decode<128>(const void*, const void*, const void*, const float*, const float*, float*,
                                        void*, int, int, int, int, cudaStream_t);

}  // namespace gdn

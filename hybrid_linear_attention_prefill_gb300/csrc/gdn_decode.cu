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
// per state row, so it is bound by HBM bandwidth: one warp per state row, each
// lane holding dk / 32 consecutive state elements (16-byte loads and stores for
// dk = 128), the two row reductions by warp shuffles.  Tensor cores would not
// help a matrix-vector step.
#include "gdn_common.cuh"

namespace gdn {

namespace {
constexpr int kDecodeWarps = 8;
constexpr int kRowsPerCta = 32;  // 4 rows per warp, processed together for ILP
}  // namespace

template <int DK>
__global__ void __launch_bounds__(32 * kDecodeWarps)
gdn_decode_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                  const __nv_bfloat16* __restrict__ v, const float* __restrict__ g,
                  const float* __restrict__ beta, float* __restrict__ state, __nv_bfloat16* __restrict__ out,
                  int Hk, int Hv, int DV) {
  constexpr int E = DK / 32;  // state elements per lane
  constexpr int R = kRowsPerCta / kDecodeWarps;
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

  const int row0 = blockIdx.y * kRowsPerCta + warp * R;
  float sv[R][E];
  float* srow[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    srow[r] = state + ((size_t)bh * DV + row0 + r) * DK + lane * E;
    if constexpr (E == 4) {
      const float4 x = *reinterpret_cast<const float4*>(srow[r]);
      sv[r][0] = x.x; sv[r][1] = x.y; sv[r][2] = x.z; sv[r][3] = x.w;
    } else if constexpr (E == 2) {
      const float2 x = *reinterpret_cast<const float2*>(srow[r]);
      sv[r][0] = x.x; sv[r][1] = x.y;
    } else {
      sv[r][0] = srow[r][0];
    }
  }
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
    if constexpr (E == 4) {
      *reinterpret_cast<float4*>(srow[r]) = make_float4(sv[r][0], sv[r][1], sv[r][2], sv[r][3]);
    } else if constexpr (E == 2) {
      *reinterpret_cast<float2*>(srow[r]) = make_float2(sv[r][0], sv[r][1]);
    } else {
      srow[r][0] = sv[r][0];
    }
    if (lane == 0) out[(size_t)bh * DV + row0 + r] = __float2bfloat16_rn(sq[r] * scale);
  }
}

template <int DK>
cudaError_t launch_decode(const void* q, const void* k, const void* v, const float* g, const float* beta,
                          float* state, void* out, int B, int Hk, int Hv, int DV, cudaStream_t st) {
  dim3 grid((unsigned)B * Hv, DV / kRowsPerCta);
  gdn_decode_kernel<DK><<<grid, 32 * kDecodeWarps, 0, st>>>(
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

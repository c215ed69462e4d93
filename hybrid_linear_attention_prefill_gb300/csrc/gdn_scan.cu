// Two-level chunk scan for long prompts with few heads (sm_103a).
//
// Within one (sequence, value head) every row s of the state evolves by the same
// affine map: with the row-vector form s_t = a_t s_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T
// of S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T (the recurrence of the
// "chunked Gated DeltaNet prefill", "Open-Jev-27B-v1.1 native text worker" page,
// "Validation and optimization scope"), a stretch of tokens maps a start state
// to S_end = S_start Phi + N.  Phi is that stretch's product of the
// a_t (I - b_t k_t k_t^T); N is the end state reached from a zero start.  So a
// long sequence is cut into P segments (on 64-token chunk boundaries), and:
//
//   pass A  every segment runs the chunk-sequential state carry twice, at once:
//           from its start state (the true initial state for segment 0, zero for
//           the others) giving N_p, and with v = 0 from the identity giving Phi_p;
//   combine S_start(1) = N_0,  S_start(p + 1) = S_start(p) Phi_p + N_p   (this file);
//   pass C  every segment runs again from S_start(p), giving the outputs and, for
//           the last segment, the final state.
//
// Passes A and C are the ordinary state-carry kernel run on the segments as packed
// sequences; this file holds the segment set-up and the fp32 combine.  The serial
// depth drops from T / 64 chunk steps to about 2 T / (64 P), at about three times
// the state-carry work -- a gain when the unsegmented problem leaves most SMs idle.
#include "gdn_common.cuh"

namespace gdn {

namespace {
constexpr int kSegThreads = 256;
constexpr int kSetupSplit = 8;    // CTAs per (segment, head) in the set-up
constexpr int kCombineRows = 4;   // state rows per combine CTA
constexpr int kCombineThreads = 128;
}  // namespace

// Segment boundaries, their chunk slots, and the two start-state sets of pass A.
//   cu_seg[i] = b T + min(p L, T) for i = b P + p (i = B P gives B T), L = chunks_per_seg * 64;
//   off_seg[i] = b nc + min(p chunks_per_seg, nc): the slot of the segment's first chunk in
//                the unsegmented (dense) chunk numbering the preparation kernel used;
//   a_init[(b P + p, h)] = init[(b, h)] for p = 0 (zeros without init), zeros otherwise;
//   i_init[(b P + p, h)] = the dk x dk identity.
// grid: (B * P * Hv, kSetupSplit); each CTA writes one row band of both states.
__global__ void __launch_bounds__(kSegThreads)
gdn_seg_setup_kernel(const float* __restrict__ init, float* __restrict__ a_init, float* __restrict__ i_init,
                     int32_t* __restrict__ cu_seg, int32_t* __restrict__ off_seg, int B, int T, int P,
                     int chunks_per_seg, int Hv, int DV, int DK) {
  const int seg = blockIdx.x / Hv, h = blockIdx.x - seg * Hv;
  const int b = seg / P, p = seg - b * P;
  const size_t n_s = (size_t)DV * DK, n_i = (size_t)DK * DK;
  {
    const size_t lo = n_s / 4 * blockIdx.y / kSetupSplit, hi = n_s / 4 * (blockIdx.y + 1) / kSetupSplit;
    float4* dst = reinterpret_cast<float4*>(a_init + ((size_t)seg * Hv + h) * n_s);
    const float4* src = (p == 0 && init != nullptr)
                            ? reinterpret_cast<const float4*>(init + ((size_t)b * Hv + h) * n_s)
                            : nullptr;
    for (size_t e = lo + threadIdx.x; e < hi; e += kSegThreads)
      dst[e] = src != nullptr ? src[e] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  {
    const size_t lo = n_i * blockIdx.y / kSetupSplit, hi = n_i * (blockIdx.y + 1) / kSetupSplit;
    float* id = i_init + ((size_t)seg * Hv + h) * n_i;
    for (size_t e = lo + threadIdx.x; e < hi; e += kSegThreads) id[e] = (e / DK == e % DK) ? 1.f : 0.f;
  }
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    const long long seg_len = (long long)chunks_per_seg * kChunk;
    const int nc = (T + kChunk - 1) / kChunk;
    for (int i = threadIdx.x; i <= B * P; i += kSegThreads) {
      const int bb = i / P, pp = i - bb * P;
      const long long off = (long long)pp * seg_len;
      const long long c0 = (long long)pp * chunks_per_seg;
      cu_seg[i] = (int32_t)((long long)bb * T + (off < T ? off : T));
      off_seg[i] = (int32_t)((long long)bb * nc + (c0 < nc ? c0 : nc));
    }
  }
}

// c_init[(b P + p, h)] = S_start(p): the initial state for p = 0, N_0 for p = 1, then
// S_start(p + 1) = S_start(p) Phi_p + N_p in fp32.  One CTA per (b, h, 4-row slice);
// thread j forms column j of the 4 rows.  The transitions Phi_p do not depend on the
// recurrence, so each goes into shared memory whole (cp.async, two buffers of DK x DK) while
// the one before it is applied: one load latency for the whole combine instead of one per tile.
// grid: (B * Hv, DV / 4); dynamic shared memory 2 DK DK floats.
__global__ void __launch_bounds__(kCombineThreads)
gdn_seg_combine_kernel(const float* __restrict__ init, const float* __restrict__ n_fin,
                       const float* __restrict__ phi, float* __restrict__ c_init, int B, int P, int Hv, int DV,
                       int DK) {
  __shared__ __align__(16) float srow[kCombineRows][128];
  extern __shared__ __align__(16) float phis[];  // [2][DK][DK]
  const int b = blockIdx.x / Hv, h = blockIdx.x - b * Hv;
  const int r0 = blockIdx.y * kCombineRows;
  const int j = threadIdx.x;
  const bool col = j < DK;
  const size_t n_s = (size_t)DV * DK, n_i = (size_t)DK * DK;
  auto state = [&](const float* base, int p) { return base + (((size_t)b * P + p) * Hv + h) * n_s; };
  auto state_out = [&](int p) { return c_init + (((size_t)b * P + p) * Hv + h) * n_s; };
  // S_start(0)
  {
    const float* src = init != nullptr ? init + ((size_t)b * Hv + h) * n_s : nullptr;
#pragma unroll
    for (int r = 0; r < kCombineRows; ++r)
      if (col) state_out(0)[(size_t)(r0 + r) * DK + j] = src != nullptr ? src[(size_t)(r0 + r) * DK + j] : 0.f;
  }
  if (P < 2) return;
  // S_start(1) = N_0
#pragma unroll
  for (int r = 0; r < kCombineRows; ++r) {
    const float x = col ? state(n_fin, 0)[(size_t)(r0 + r) * DK + j] : 0.f;
    srow[r][j] = x;
    if (col) state_out(1)[(size_t)(r0 + r) * DK + j] = x;
  }
  // Phi_p (p = 1 .. P - 2) into buffer p & 1
  auto load_phi = [&](int p) {
    const float* ph = phi + (((size_t)b * P + p) * Hv + h) * n_i;
    float* dst = phis + (size_t)(p & 1) * n_i;
    for (size_t e = threadIdx.x; e < n_i / 4; e += kCombineThreads) cp_async16(dst + 4 * e, ph + 4 * e, true);
    cp_async_commit();
  };
  // N_p's rows of this CTA, a segment ahead (they do not depend on the recurrence either)
  float nxt[kCombineRows];
  auto load_n = [&](int p) {
    const float* nf = state(n_fin, p);
#pragma unroll
    for (int u = 0; u < kCombineRows; ++u) nxt[u] = col ? nf[(size_t)(r0 + u) * DK + j] : 0.f;
  };
  if (P > 2) {
    load_phi(1);
    load_n(1);
  }
  for (int p = 1; p + 1 < P; ++p) {
    const bool next = p + 2 < P;
    if (next) load_phi(p + 1);  // into the other buffer, read last at p - 1 (barrier below)
    float acc[kCombineRows];
#pragma unroll
    for (int u = 0; u < kCombineRows; ++u) acc[u] = nxt[u];
    if (next) load_n(p + 1);
    if (next) cp_async_wait<1>();
    else cp_async_wait<0>();
    __syncthreads();  // Phi_p, and the previous rows in srow, visible
    if (col) {  // the rows' entries four at a time (16-byte broadcast loads), in order
      const float* f = phis + (size_t)(p & 1) * n_i + j;
#pragma unroll 2
      for (int kk = 0; kk < DK; kk += 4) {
        const float f0 = f[(size_t)kk * DK], f1 = f[(size_t)(kk + 1) * DK], f2 = f[(size_t)(kk + 2) * DK],
                    f3 = f[(size_t)(kk + 3) * DK];
#pragma unroll
        for (int u = 0; u < kCombineRows; ++u) {
          const float4 sv = *reinterpret_cast<const float4*>(&srow[u][kk]);
          acc[u] = fmaf(sv.x, f0, acc[u]);
          acc[u] = fmaf(sv.y, f1, acc[u]);
          acc[u] = fmaf(sv.z, f2, acc[u]);
          acc[u] = fmaf(sv.w, f3, acc[u]);
        }
      }
    }
    __syncthreads();  // Phi_p and srow read before they are overwritten
#pragma unroll
    for (int u = 0; u < kCombineRows; ++u) {
      srow[u][j] = acc[u];
      if (col) state_out(p + 1)[(size_t)(r0 + u) * DK + j] = acc[u];
    }
  }
}

cudaError_t launch_seg_setup(const float* init, float* a_init, float* i_init, int32_t* cu_seg, int32_t* off_seg,
                             int B, int T, int P, int chunks_per_seg, int Hv, int DV, int DK, cudaStream_t st) {
  dim3 grid((unsigned)(B * P * Hv), kSetupSplit);
  gdn_seg_setup_kernel<<<grid, kSegThreads, 0, st>>>(init, a_init, i_init, cu_seg, off_seg, B, T, P,
                                                     chunks_per_seg, Hv, DV, DK);
  return cudaGetLastError();
}

cudaError_t launch_seg_combine(const float* init, const float* n_fin, const float* phi, float* c_init, int B,
                               int P, int Hv, int DV, int DK, cudaStream_t st) {
  const int smem = 2 * DK * DK * (int)sizeof(float);  // 128 KB at dk = 128
  cudaError_t e = set_smem_limit_once<gdn_seg_combine_kernel>(2 * 128 * 128 * (int)sizeof(float));
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(B * Hv), (unsigned)(DV / kCombineRows));
  gdn_seg_combine_kernel<<<grid, kCombineThreads, smem, st>>>(init, n_fin, phi, c_init, B, P, Hv, DV, DK);
  return cudaGetLastError();
}

}  // namespace gdn

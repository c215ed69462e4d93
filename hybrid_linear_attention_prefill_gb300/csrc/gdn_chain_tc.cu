// Chunk-sequential state carry on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// One CTA of 8 warps owns a 16-, 32- or 64-row slice of the dv x dk state S of one
// (sequence, value head) and walks the sequence's 64-token chunks in order.
// For a chunk starting from S (rows beyond the chunk's n tokens are zero,
// with g = beta = 0), with Tm = (I + A)^-1 and PT = P Tm from the preparation
// kernel, gamma = cumsum(g), e = exp(gamma), d = exp(gamma_last - gamma):
//
//   phase 1   [X; Y] = [K; Q] S^T                       (M = 128 stacked tokens, K = dk)
//             R      = diag(beta) V - diag(beta e) X
//   phase 2   [U; Z] = [Tm; PT] R                       (M = 128, K = 64)
//             O      = scale (diag(e) Y + Z)            -> bf16 outputs
//   phase 3   dS^T   = K^T diag(d) U                    (M = dk = 128, K = 64)
//             S      = e_last S + dS
//
// which is the chunk form of S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T,
// o_t = S_t q_t / sqrt(dk) (the "chunked Gated DeltaNet prefill" of the
// "Open-Jev-27B-v1.1 native text worker" page, "Validation and optimization
// scope").
//
// Latency, not arithmetic, bounds this loop.  On sm_103a one thread issues a
// tcgen05.mma of M = 64 or 128 and N <= 64 every ~45 cycles, whether or not it
// accumulates into the previous one's accumulator, and the result is visible
// ~60 cycles after the last issue; at N = 64 the tensor math itself would take
// ~37 cycles.  So
//  * the operand that carries the state in each phase (S, R, diag(d) U) is
//    split into bf16 hi and lo parts that are stacked along N (N = 64: columns
//    0..31 hi, 32..63 lo) instead of being issued as two MMAs, keeping the fp32
//    state accurate to ~2^-16 at no extra MMA;
//  * phase 1 splits its K = dk steps over two TMEM accumulators, phases 2 and 3
//    use one (64 columns each, 128 allocated): each extra accumulator costs the
//    epilogue another 32-column TMEM read per thread, and measured, two in
//    phase 1 and one in phases 2-3 is fastest.
// A ninth warp only issues: the MMAs of each phase (ending with a tcgen05.commit
// on an mbarrier) and the TMA loads two chunks ahead (K, Q, the value slice and
// the [Tm; PT] tile: 5-6 bulk-tensor copies into a ring of three stages).  A
// chunk's copies take about a microsecond to land under the load of all CTAs,
// about half a chunk step, so one stage ahead would leave them on the critical
// path.
// Epilogue warps w and w + 4 read the same 32 TMEM lanes (rows) and split the
// 32 state columns between them.  The state S stays in fp32 registers.
//
// Shared-memory layouts (tile bases 1024-byte aligned):
//   [K; Q]   K-major, 128 B swizzle: [dk/64 blocks][128 rows][128 B]; rows 0..63 K, 64..127 Q.
//            The same K rows, read MN-major (dk contiguous), are phase 3's A operand.
//   [Tm; PT] K-major, 128 B swizzle: [128 rows][128 B].
//   S, R, U  MN-major, 128 B swizzle: one row per K index (d or token), 128 B =
//            for each half of the 32 slice columns, 16 bf16 hi parts then 16 lo parts.
//   V        the 32-column value slice, 64 B rows, 64 B swizzle.
// TMA writes these layouts directly; out-of-range box elements (tokens past
// the end, d >= dk) arrive as zeros.
#include "gdn_tc.cuh"
#include "gdn_tmap.cuh"

namespace gdn {

namespace {

constexpr int kThreads = 288;   // 8 epilogue warps + 1 issue warp
constexpr int kEpiThreads = 256;
constexpr int kParts = 2;       // accumulators in phase 1 (K = dk)
constexpr int kParts23 = 1;     // and in phases 2 and 3 (K = 64)
constexpr uint32_t kMaxPolls = 1u << 24;

// Layout of a CTA that owns DVT = 16, 32 or 64 rows of the state.  The MMAs carry the bf16 hi
// and lo parts of the slice along N = 2 DVT.  A 128-byte swizzle atom of an MN-major operand row
// holds 64 bf16 = 32 state columns (16 hi, 16 lo per 16-column group), so the DVT = 64 operands
// are two atoms wide, the second one atom's bytes after the first (the descriptor's leading byte
// offset), and the DVT = 16 ones use the first 32 columns (before the swizzle) of each row.
template <int DVT>
struct Cfg {
  static constexpr int kN = 2 * DVT;
  static constexpr int kAtoms = (kN + 63) / 64;
  static constexpr int kGroups = DVT / 32;            // 16-column groups per epilogue thread (16 rows: half of one)
  static constexpr uint32_t kTmemCols = kParts * kN;   // phase 1's partial accumulators
  // stage layout (bytes)
  static constexpr int kOffKQ = 0;                  // 2 x 16384
  static constexpr int kOffTP = 32768;              // 16384
  static constexpr int kOffV = kOffTP + 16384;      // 64 rows x 2 DVT bytes (none / 64 / 128 B swizzle)
  static constexpr int kVBytes = 64 * 2 * DVT;
  static constexpr int kOffG = kOffV + kVBytes;     // 64 fp32
  static constexpr int kOffB = kOffG + 256;         // 64 fp32
  static constexpr int kOffRN = kOffB + 256;        // 128 fp32: inverse norms of the k rows, then the q rows
  static constexpr int kStage = (kOffRN + 512 + 1023) / 1024 * 1024;  // 51, 53, 57 KB (16, 32, 64 rows)
  // TMA ring: chunk c + kStages - 1 loads during chunk c (two ahead with 16 and 32 rows; 64 rows
  // leave room for two stages, so one ahead)
  static constexpr int kStages = DVT == 64 ? 2 : 3;
  // B operands after the stages: S (dk rows), R and dU (64 token rows), kAtoms atoms each
  static constexpr int kAtomS = 128 * 128, kAtomRU = 64 * 128;
  static constexpr int kOffS = kStages * kStage;
  static constexpr int kOffR = kOffS + kAtoms * kAtomS;
  static constexpr int kOffU = kOffR + kAtoms * kAtomRU;
  // 64 rows: the Y rows of the output warps wait here between phases 1 and 2 ([32 columns][128 threads])
  static constexpr int kOffY = kOffU + kAtoms * kAtomRU;
  static constexpr int kYBytes = DVT == 64 ? 32 * 128 * 4 : 0;
  static constexpr int kOffBar = kOffY + kYBytes;  // 3 MMA mbarriers, the load mbarriers, TMEM base, abort flag
  static constexpr int kSmemBytes = kOffBar + 64 + 1024;   // + slack for 1024-byte alignment
  static constexpr uint32_t kID_KS = tc::idesc_bf16(128, kN, 0, 1);  // A K-major, B MN-major
  static constexpr uint32_t kID_KT = tc::idesc_bf16(128, kN, 1, 1);  // A MN-major, B MN-major
  static_assert(DVT == 16 || DVT == 32 || DVT == 64, "16, 32 or 64 state rows per CTA");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert((3 + kStages) * 8 <= 48, "mbarriers in the barrier block");
};

// Write 16 fp32 values (state columns 16 g .. 16 g + 15) of one operand row as bf16 hi parts and
// lo parts: group g sits in swizzle atom g / 2 (atom_bytes apart), hi in 16-byte chunks
// 4 (g % 2), + 1 and lo in + 2, + 3, so that accumulator columns 32 g .. 32 g + 31 hold this
// group's hi then lo sums.
__device__ __forceinline__ void store_split16(unsigned char* tile, int atom_bytes, uint32_t row, int g,
                                              const float* x) {
  tile += (g >> 1) * atom_bytes;
  const int c = 4 * (g & 1);
  uint32_t h[8], l[8];
#pragma unroll
  for (int p = 0; p < 8; ++p) split_bf16(x[2 * p], x[2 * p + 1], h[p], l[p]);
  *reinterpret_cast<uint4*>(tile + tc::sw128(row, c)) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(tile + tc::sw128(row, c + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
  *reinterpret_cast<uint4*>(tile + tc::sw128(row, c + 2)) = make_uint4(l[0], l[1], l[2], l[3]);
  *reinterpret_cast<uint4*>(tile + tc::sw128(row, c + 3)) = make_uint4(l[4], l[5], l[6], l[7]);
}

// 16-row CTAs: a thread owns 8 of the group's 16 columns, h = 0 or 1.  Its hi parts are 16-byte
// chunk h of the operand row, its lo parts chunk 2 + h.
__device__ __forceinline__ void store_split8(unsigned char* tile, uint32_t row, int h, const float* x) {
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) split_bf16(x[2 * p], x[2 * p + 1], hi[p], lo[p]);
  *reinterpret_cast<uint4*>(tile + tc::sw128(row, h)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint4*>(tile + tc::sw128(row, 2 + h)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// acc[i] = sum over the NP partials (N columns apart) of the hi and lo products of state column
// 8 h + i: hi in accumulator column 8 h + i, lo in 16 + 8 h + i.
template <int NP, int N>
__device__ __forceinline__ void sum_parts8(uint32_t taddr, int h, float (&acc)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    float hi[8], lo[8];
    tc::tmem_ld8(taddr + N * p + 8 * h, hi);
    tc::tmem_ld8(taddr + N * p + 16 + 8 * h, lo);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += hi[i] + lo[i];
  }
}

// acc[i] = sum over the NP partial accumulators (N columns apart) of the hi and lo products of
// state column 16 g + i (partial p holds columns N p + 32 g ..: 16 hi, 16 lo).  With N = 64 two
// partials are read by one TMEM load; with N = 128 one at a time, to hold fewer registers.
template <int NP, int N>
__device__ __forceinline__ void sum_parts(uint32_t taddr, int g, float (&acc)[16]) {
  if constexpr (NP == 2 && N == 64) {
    float t[64];
    tc::tmem_ld32x2(taddr + 32 * g, taddr + N + 32 * g, t);
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = (t[i] + t[16 + i]) + (t[32 + i] + t[48 + i]);
  } else {
    float t[32];
    tc::tmem_ld32(taddr + 32 * g, t);
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = t[i] + t[16 + i];
#pragma unroll
    for (int p = 1; p < NP; ++p) {
      tc::tmem_ld32(taddr + N * p + 32 * g, t);
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] += t[i] + t[16 + i];
    }
  }
}

}  // namespace

// kNorm: q and k are normalised in-kernel (their inverse norms come from the
// preparation kernel); a separate instantiation keeps the plain path free of it.
// One CTA per SM.  Nine warps leave three on one of the SM's four sub-partitions, whose 16 K
// registers then cap a thread at 168: the 64-row slice reads its partial sums 32 columns at a
// time to stay within it.
template <int DK, bool kNorm, int DVT>
__global__ void __launch_bounds__(kThreads, 1)
gdn_chain_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
                    const float* __restrict__ g, const float* __restrict__ beta, const int32_t* __restrict__ cu,
                    const int32_t* __restrict__ chunk_off, const int32_t* __restrict__ order,
                    const float* __restrict__ ws_rn, const float* init,
                    __nv_bfloat16* __restrict__ out,
                    float* fin, int* __restrict__ err, int B, int T, int Hk, int Hv, int DV, int nc_dense,
                    long long nslots, int h_base, int c_begin, int c_end) {
  // Launched as a programmatic dependent of the kernel before it in the stream (the preparation
  // kernel): the CTA starts while that kernel's last CTAs run and waits here until it has
  // completed and its writes are visible (otherwise this returns at once).
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  using C = Cfg<DVT>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t pad = ((raw_s + 1023u) & ~1023u) - raw_s;
  unsigned char* sm = smem_raw + pad;
  const uint32_t sb = raw_s + pad;  // shared-window address of sm

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);     // [0..2] MMA phases
  uint64_t* full = bars + 3;                                          // [0..kStages) stage loaded
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffBar + 48);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kOffBar + 52);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool issuer = warp == 8;
  const int q4 = warp & 3;         // TMEM lane quadrant (epilogue warps)
  const int half = (warp >> 2) & 1;  // state columns 16 g .. 16 g + 15 for g = kGroups half + gg
  const int row = 32 * q4 + lane;
  const int ntiles = DV / DVT;
  // CTA (x, y) = (sequence b x slices + slice, head).  With a dispatch order (packed batches),
  // the CTA's position in dispatch order walks the sequences most chunks first, and every
  // head and slice of one sequence before the next, so that the long chains start first.
  int bx = (int)blockIdx.x, hy = (int)blockIdx.y;
  if (order != nullptr) {
    const long long pos = (long long)blockIdx.y * gridDim.x + blockIdx.x;
    const int per = (int)gridDim.y * ntiles;  // CTAs of one sequence
    const int r = (int)(pos / per), rem = (int)(pos - (long long)r * per);
    const int ob = order[r];
    hy = rem / ntiles;
    bx = (ob >= 0 && ob < B ? ob : r) * ntiles + rem % ntiles;
  }
  const int b = bx / ntiles;
  const int dv0 = (bx - b * ntiles) * DVT;
  const int h = h_base + hy;
  const int hk = h / (Hv / Hk);
  const float scale = rsqrtf((float)DK);
  constexpr int kP1 = DK / 16 < kParts ? DK / 16 : kParts;  // partials used by phase 1
  constexpr int kKBlocks = DK > 64 ? 2 : 1;                  // 64-wide d blocks loaded per tile
  constexpr uint32_t kTxBytes = 2 * kKBlocks * 8192 + C::kVBytes + 16384;
  constexpr int kAhead = C::kStages - 1;  // chunks whose tiles are in flight ahead of the current one

  const SeqChunk sq = seq_bounds(cu, b, T);
  const int slot0 = cu == nullptr ? b * nc_dense : chunk_off[b];
  int nchunks = (sq.len + kChunk - 1) / kChunk;
  if ((long long)slot0 + nchunks > nslots) nchunks = slot0 < nslots ? (int)(nslots - slot0) : 0;
  // this launch walks chunks c0 .. c1 - 1 of the sequence, from `init` (the state before
  // chunk c0) to `fin` (the state after chunk c1 - 1): the whole sequence, or a window of
  // it whose neighbours run as other launches in order
  const int c0 = c_begin < nchunks ? c_begin : nchunks;
  const int c1 = c_end < nchunks ? c_end : nchunks;

  // ---- set-up: TMEM, barriers, zero d-block 1 when dk <= 64 --------------------
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, C::kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 3 + C::kStages; ++i) tc::mbar_init(&bars[i], 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (issuer && lane == 0) {
    tc::prefetch_tensormap(&tm_k);
    tc::prefetch_tensormap(&tm_q);
    tc::prefetch_tensormap(&tm_v);
    tc::prefetch_tensormap(&tm_w);
  }
  if (kKBlocks == 1 && !issuer) {  // phase 3 reads all 128 rows of K^T: the rows d >= 64 stay zero
    for (int e = tid; e < C::kStages * 1024; e += kEpiThreads) {
      const int stg = e >> 10, w = e & 1023;
      *reinterpret_cast<uint4*>(sm + stg * C::kStage + C::kOffKQ + 16384 + w * 16) = make_uint4(0, 0, 0, 0);
    }
  }

  // ---- initial state: thread (row d, half) holds S[16 g + i][d], g = kGroups half + gg ----
  // (16 rows: S[8 half + i][d])
  const int d = row;
  constexpr int kCols = DVT / 2;  // state columns per epilogue thread
  float s[kCols];
  if (!issuer && DVT == 16) {
    const size_t base = ((size_t)b * Hv + h) * DV + dv0 + 8 * half;
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = (init != nullptr && d < DK) ? init[(base + i) * DK + d] : 0.f;
    store_split8(sm + C::kOffS, d, half, s);
  }
  if (!issuer) {
#pragma unroll
    for (int gg = 0; gg < C::kGroups; ++gg) {
      const int g = C::kGroups * half + gg;
      const size_t base = ((size_t)b * Hv + h) * DV + dv0 + 16 * g;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        s[16 * gg + i] = (init != nullptr && d < DK) ? init[(base + i) * DK + d] : 0.f;
      store_split16(sm + C::kOffS, C::kAtomS, d, g, s + 16 * gg);
    }
  }
  tc::fence_proxy_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tq = tmem + ((uint32_t)(32 * q4) << 16);  // this warp's lanes

  // TMA for the tiles of chunk c into stage stg (one thread); g and beta by cp.async.
  auto load_tiles = [&](int c, int stg) {
    unsigned char* st = sm + stg * C::kStage;
    const int t0 = (int)(sq.bos + (long long)c * kChunk);
    tc::mbar_arrive_expect_tx(&full[stg], kTxBytes);
#pragma unroll
    for (int db = 0; db < kKBlocks; ++db) {
      tc::tma_load_3d(st + C::kOffKQ + db * 16384, &tm_k, 64 * db, hk, t0, &full[stg]);
      tc::tma_load_3d(st + C::kOffKQ + db * 16384 + 8192, &tm_q, 64 * db, hk, t0, &full[stg]);
    }
    tc::tma_load_3d(st + C::kOffV, &tm_v, dv0, h, t0, &full[stg]);
    tc::tma_load_2d(st + C::kOffTP, &tm_w, 0, (int)(((long long)(slot0 + c) * Hv + h) * 128), &full[stg]);
  };
  auto load_scalars = [&](int c, int stg) {
    unsigned char* st = sm + stg * C::kStage;
    if (tid < kChunk) {
      const int n = min(kChunk, sq.len - c * kChunk);
      const bool ok = tid < n;
      const size_t off = ok ? (size_t)(sq.bos + (long long)c * kChunk + tid) * Hv + h : 0;
      cp_async4(st + C::kOffG + 4 * tid, g + off, ok);
      cp_async4(st + C::kOffB + 4 * tid, beta + off, ok);
      if (kNorm) {  // the chunk's inverse norms, from the preparation kernel
        const float* rn = ws_rn + ((size_t)(slot0 + c) * Hk + hk) * (2 * kChunk);
        cp_async4(st + C::kOffRN + 4 * tid, rn + tid, true);
        cp_async4(st + C::kOffRN + 256 + 4 * tid, rn + kChunk + tid, true);
      }
    }
  };

  if (c1 > c0) {
    if (issuer && lane == 0)
      for (int a = 0; a < kAhead && c0 + a < c1; ++a) load_tiles(c0 + a, a);
    load_scalars(c0, 0);
  }
  cp_async_commit();

  const int tok = 32 * (q4 & 1) + lane;  // this thread's token in phases 1-2
  bool aborted = false;
  int c = c0;
  for (; c < c1; ++c) {
    const int ci = c - c0;  // position in this launch: stage and barrier phases
    const int stg = ci % C::kStages;
    const uint32_t par = (uint32_t)(ci & 1);
    unsigned char* st = sm + stg * C::kStage;
    const uint32_t st_s = sb + stg * C::kStage;
    cp_async_wait<0>();
    // The thread that issued the stage's copies waits for them; the barrier publishes them to
    // every thread.  All threads read the abort flag right after each barrier (so they leave the
    // loop at the same one); the issuing thread acts on it after issuing that phase's MMAs.
    if (issuer && lane == 0 && !tc::mbar_wait(&full[stg], (uint32_t)((ci / C::kStages) & 1), kMaxPolls)) {
      *abort_flag = 1;
      atomicOr(err, 2);
    }
    __syncthreads();
    const int ab_top = *abort_flag;

    if (issuer) {
      // ---- phase 1: [X; Y] = [K; Q] [S_hi | S_lo]^T --------------------------------
      if (lane == 0) {
        tc::fence_after();
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks) {
          const uint64_t a = tc::sdesc(st_s + C::kOffKQ + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024, tc::kSw128);
          const uint64_t bd = tc::sdesc(sb + C::kOffS + ks * 2048, C::kAtomS, 1024, tc::kSw128);
          tc::mma_bf16(tmem + C::kN * (ks % kP1), a, bd, C::kID_KS, ks >= kP1);
        }
        tc::commit(&bars[0]);
        // stage (ci + kAhead) % kStages = (ci - 1) % kStages was last read by the previous
        // chunk's MMAs, which are done
        if (c + kAhead < c1) load_tiles(c + kAhead, (ci + kAhead) % C::kStages);
      }
      __syncwarp();
      if (ab_top) { aborted = true; break; }
      __syncthreads();  // R written
      const int ab_r = *abort_flag;
      // ---- phase 2: [U; Z] = [Tm; PT] [R_hi | R_lo] --------------------------------
      if (lane == 0) {
        tc::fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t a = tc::sdesc(st_s + C::kOffTP + ks * 32, 16, 1024, tc::kSw128);
          const uint64_t bd = tc::sdesc(sb + C::kOffR + ks * 2048, C::kAtomRU, 1024, tc::kSw128);
          tc::mma_bf16(tmem + C::kN * (ks % kParts23), a, bd, C::kID_KS, ks >= kParts23);
        }
        tc::commit(&bars[1]);
      }
      __syncwarp();
      if (ab_r) { aborted = true; break; }
      __syncthreads();  // dU written
      const int ab_d = *abort_flag;
      // ---- phase 3: dS^T = K^T [dU_hi | dU_lo] -------------------------------------
      if (lane == 0) {
        tc::fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t a = tc::sdesc(st_s + C::kOffKQ + ks * 2048, 16384, 1024, tc::kSw128);
          const uint64_t bd = tc::sdesc(sb + C::kOffU + ks * 2048, C::kAtomRU, 1024, tc::kSw128);
          tc::mma_bf16(tmem + C::kN * (ks % kParts23), a, bd, C::kID_KT, ks >= kParts23);
        }
        tc::commit(&bars[2]);
      }
      __syncwarp();
      if (ab_d) { aborted = true; break; }
      continue;
    }

    // ================= epilogue warps =================
    if (ab_top) { aborted = true; break; }
    if (c + 1 < c1) load_scalars(c + 1, (ci + 1) % C::kStages);
    cp_async_commit();

    // per-token scalars: every warp scans the 64 log decays of the chunk
    const float* gs = reinterpret_cast<const float*>(st + C::kOffG);
    const float* bs = reinterpret_cast<const float*>(st + C::kOffB);
    float g0 = gs[lane], g1 = gs[lane + 32];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u0 = __shfl_up_sync(0xffffffffu, g0, o);
      const float u1 = __shfl_up_sync(0xffffffffu, g1, o);
      if (lane >= o) { g0 += u0; g1 += u1; }
    }
    g1 += __shfl_sync(0xffffffffu, g0, 31);
    const float glast = __shfl_sync(0xffffffffu, g1, 31);
    const float gam = (q4 & 1) ? g1 : g0;
    const float e_t = expf(gam);
    const float d_t = expf(glast - gam);
    const float eC = expf(glast);
    const float b_t = bs[tok];
    // with in-kernel q/k normalisation, this token's inverse norm (k rows for the
    // R / dU epilogues, q rows for the outputs), as the preparation kernel summed it
    const float rn = kNorm ? reinterpret_cast<const float*>(st + C::kOffRN)[tok + (q4 < 2 ? 0 : 64)] : 1.f;

    // ---- phase-1 epilogue: R = beta V - beta e X (rows 0..63), keep Y (rows 64..127)
    if (!tc::mbar_wait(&bars[0], par, kMaxPolls)) { *abort_flag = 1; atomicOr(err, 1); }
    tc::fence_after();
    // Y rows of the output warps (q4 >= 2) until phase 2: 32 rows keep their one group in registers,
    // 64 rows their two groups in shared memory (column-major over the 128 output threads)
    float acc[16], y[1][16];
    float* ys = reinterpret_cast<float*>(sm + C::kOffY) + (q4 >= 2 ? 32 * (q4 - 2) + lane + 64 * half : 0);
    if constexpr (DVT == 16) {  // 8 columns a thread: value bytes 16 half of the 32-byte row
      float a8[8];
      sum_parts8<kP1, C::kN>(tq, half, a8);
      if (q4 < 2) {
        const float be = b_t * e_t * rn;
        const uint4 raw = *reinterpret_cast<const uint4*>(st + C::kOffV + tok * 32 + 16 * half);
        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float2 vv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[p]));
          a8[2 * p] = b_t * vv.x - be * a8[2 * p];
          a8[2 * p + 1] = b_t * vv.y - be * a8[2 * p + 1];
        }
        store_split8(sm + C::kOffR, tok, half, a8);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) y[0][i] = a8[i] * rn;
      }
    }
#pragma unroll
    for (int gg = 0; gg < C::kGroups; ++gg) {
      const int g = C::kGroups * half + gg;
      sum_parts<kP1, C::kN>(tq, g, acc);
      if (q4 < 2) {
        const unsigned char* vrow = st + C::kOffV;
        const float be = b_t * e_t * rn;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // the group's two 16-byte chunks of the value row
          uint32_t voff;
          if constexpr (DVT == 32) voff = tc::sw64(tok, 2 * g + hh);
          else voff = tc::sw128(tok, 2 * g + hh);
          const uint4 raw = *reinterpret_cast<const uint4*>(vrow + voff);
          const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const float2 vv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[p]));
            const int i = 8 * hh + 2 * p;
            acc[i] = b_t * vv.x - be * acc[i];
            acc[i + 1] = b_t * vv.y - be * acc[i + 1];
          }
        }
        store_split16(sm + C::kOffR, C::kAtomRU, tok, g, acc);
      } else if constexpr (DVT == 32) {
#pragma unroll
        for (int i = 0; i < 16; ++i) y[gg][i] = acc[i] * rn;
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) ys[(16 * gg + i) * 128] = acc[i] * rn;
      }
    }
    if (q4 < 2) tc::fence_proxy_async();  // R is read by the tensor core next
    tc::fence_before();
    __syncthreads();  // R written
    if (*abort_flag) { aborted = true; break; }

    // ---- phase-2 epilogue: dU (rows 0..63); outputs from Z (rows 64..127) ------------
    if (!tc::mbar_wait(&bars[1], par, kMaxPolls)) { *abort_flag = 1; atomicOr(err, 1); }
    tc::fence_after();
    uint32_t o8[C::kGroups > 0 ? C::kGroups : 1][8];
    if constexpr (DVT == 16) {
      float a8[8];
      sum_parts8<kParts23, C::kN>(tq, half, a8);
      if (q4 < 2) {
        const float dr = d_t * rn;
#pragma unroll
        for (int i = 0; i < 8; ++i) a8[i] *= dr;
        store_split8(sm + C::kOffU, tok, half, a8);
      } else {
        const float es = scale * e_t;
#pragma unroll
        for (int p = 0; p < 4; ++p)
          o8[0][p] = pack_bf16(es * y[0][2 * p] + scale * a8[2 * p], es * y[0][2 * p + 1] + scale * a8[2 * p + 1]);
      }
    }
#pragma unroll
    for (int gg = 0; gg < C::kGroups; ++gg) {
      const int g = C::kGroups * half + gg;
      sum_parts<kParts23, C::kN>(tq, g, acc);
      if (q4 < 2) {
        const float dr = d_t * rn;
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] *= dr;
        store_split16(sm + C::kOffU, C::kAtomRU, tok, g, acc);
      } else {
        const float es = scale * e_t;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          float y0, y1;
          if constexpr (DVT == 32) { y0 = y[gg][2 * p]; y1 = y[gg][2 * p + 1]; }
          else { y0 = ys[(16 * gg + 2 * p) * 128]; y1 = ys[(16 * gg + 2 * p + 1) * 128]; }
          o8[gg][p] = pack_bf16(es * y0 + scale * acc[2 * p], es * y1 + scale * acc[2 * p + 1]);
        }
        if constexpr (DVT == 64) {  // stored now: the packed outputs do not stay live across the barrier
          const int n = min(kChunk, sq.len - c * kChunk);
          if (tok < n) {
            __nv_bfloat16* orow = out + ((size_t)(sq.bos + (long long)c * kChunk + tok) * Hv + h) * DV + dv0 + 16 * g;
            *reinterpret_cast<uint4*>(orow) = make_uint4(o8[gg][0], o8[gg][1], o8[gg][2], o8[gg][3]);
            *reinterpret_cast<uint4*>(orow + 8) = make_uint4(o8[gg][4], o8[gg][5], o8[gg][6], o8[gg][7]);
          }
        }
      }
    }
    if (q4 < 2) tc::fence_proxy_async();  // dU is read by the tensor core next
    tc::fence_before();
    __syncthreads();  // dU written
    if (*abort_flag) { aborted = true; break; }

    // outputs go out while the phase-3 MMAs run
    if (DVT == 16 && q4 >= 2) {
      const int n = min(kChunk, sq.len - c * kChunk);
      if (tok < n) {
        __nv_bfloat16* orow = out + ((size_t)(sq.bos + (long long)c * kChunk + tok) * Hv + h) * DV + dv0 + 8 * half;
        *reinterpret_cast<uint4*>(orow) = make_uint4(o8[0][0], o8[0][1], o8[0][2], o8[0][3]);
      }
    }
    if (DVT == 32 && q4 >= 2) {
      const int n = min(kChunk, sq.len - c * kChunk);
      if (tok < n) {
#pragma unroll
        for (int gg = 0; gg < C::kGroups; ++gg) {
          __nv_bfloat16* orow = out + ((size_t)(sq.bos + (long long)c * kChunk + tok) * Hv + h) * DV + dv0 +
                                16 * (C::kGroups * half + gg);
          *reinterpret_cast<uint4*>(orow) = make_uint4(o8[gg][0], o8[gg][1], o8[gg][2], o8[gg][3]);
          *reinterpret_cast<uint4*>(orow + 8) = make_uint4(o8[gg][4], o8[gg][5], o8[gg][6], o8[gg][7]);
        }
      }
    }

    // ---- phase-3 epilogue: S = e_last S + dS ------------------------------------------
    if (!tc::mbar_wait(&bars[2], par, kMaxPolls)) { *abort_flag = 1; atomicOr(err, 1); }
    tc::fence_after();
    if constexpr (DVT == 16) {
      float a8[8];
      sum_parts8<kParts23, C::kN>(tq, half, a8);
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i] = fmaf(eC, s[i], a8[i]);
      store_split8(sm + C::kOffS, d, half, s);
    }
#pragma unroll
    for (int gg = 0; gg < C::kGroups; ++gg) {
      const int g = C::kGroups * half + gg;
      sum_parts<kParts23, C::kN>(tq, g, acc);
#pragma unroll
      for (int i = 0; i < 16; ++i) s[16 * gg + i] = fmaf(eC, s[16 * gg + i], acc[i]);
      store_split16(sm + C::kOffS, C::kAtomS, d, g, s + 16 * gg);
    }
    tc::fence_proxy_async();  // S is read by the tensor core at the next chunk
    tc::fence_before();
  }

  // ---- final state, clean-up -------------------------------------------------------
  cp_async_wait<0>();
  if (!aborted && !issuer && fin != nullptr && d < DK) {
    if constexpr (DVT == 16) {
      const size_t base = ((size_t)b * Hv + h) * DV + dv0 + 8 * half;
#pragma unroll
      for (int i = 0; i < 8; ++i) fin[(base + i) * DK + d] = s[i];
    }
#pragma unroll
    for (int gg = 0; gg < C::kGroups; ++gg) {
      const size_t base = ((size_t)b * Hv + h) * DV + dv0 + 16 * (C::kGroups * half + gg);
#pragma unroll
      for (int i = 0; i < 16; ++i) fin[(base + i) * DK + d] = s[16 * gg + i];
    }
  }
  if (aborted && issuer && lane == 0) {
    // let MMAs and TMA copies still in flight land before the CTA exits (bounded again)
    const int ci = c - c0;
    const uint32_t par = (uint32_t)(ci & 1);
    for (int i = 0; i < 3; ++i) (void)tc::mbar_wait(&bars[i], par, 1u << 16);
    for (int i = 0; i < C::kStages; ++i)
      (void)tc::mbar_wait(&full[(ci + i) % C::kStages], (uint32_t)(((ci + i) / C::kStages) & 1), 1u << 16);
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, C::kTmemCols);
}

// The bounded-wait path of the kernels, run on purpose: an mbarrier that nothing
// completes, waited on with the same helper and the same give-up handling.
__global__ void gdn_wait_timeout_probe_kernel(int max_polls, int* __restrict__ status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (!tc::mbar_wait(&bar, 0, (uint32_t)max_polls)) atomicOr(status, 1);
}

cudaError_t launch_wait_timeout_probe(int max_polls, int* status, cudaStream_t st) {
  gdn_wait_timeout_probe_kernel<<<1, 32, 0, st>>>(max_polls, status);
  return cudaGetLastError();
}

namespace {

// A bf16 tiled tensor map; dims / strides listed innermost first, strides in bytes.
bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
              const cuuint32_t* box, CUtensorMapSwizzle swz) {
  return make_map16(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides, box, swz);
}

}  // namespace

template <int DK, int DVT>
cudaError_t launch_chain_tc_dvt(const CUtensorMap& mk, const CUtensorMap& mq, const void* v, const CUtensorMap& mw,
                                const float* g, const float* beta, const int32_t* cu, const int32_t* chunk_off,
                                const int32_t* order, const float* ws_rn, const float* init, void* out, float* fin,
                                int* err, int B, int T, int Hk, int Hv, int DV, int nc_dense, long long nslots,
                                int norm_qk, int h_base, int h_count, int c_begin, int c_end, cuuint64_t tt,
                                cudaStream_t st) {
  using C = Cfg<DVT>;
  CUtensorMap mv;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)DV, (cuuint64_t)Hv, tt};
    const cuuint64_t strides[2] = {(cuuint64_t)DV * 2, (cuuint64_t)Hv * DV * 2};
    const cuuint32_t box[3] = {DVT, 1, 64};
    const CUtensorMapSwizzle swz =
        DVT == 16 ? CU_TENSOR_MAP_SWIZZLE_NONE : DVT == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    if (!make_map(&mv, v, 3, dims, strides, box, swz)) return cudaErrorInvalidValue;
  }
  auto* kernel = norm_qk ? gdn_chain_tc_kernel<DK, true, DVT> : gdn_chain_tc_kernel<DK, false, DVT>;
  cudaError_t e = norm_qk ? set_smem_limit_once<gdn_chain_tc_kernel<DK, true, DVT>>(C::kSmemBytes)
                          : set_smem_limit_once<gdn_chain_tc_kernel<DK, false, DVT>>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // value heads h_base .. h_base + h_count - 1; a programmatic dependent of the kernel before it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B * (DV / DVT), h_count);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, mk, mq, mv, mw, g, beta, cu, chunk_off, order, ws_rn, init,
                         static_cast<__nv_bfloat16*>(out), fin, err, B, T, Hk, Hv, DV, nc_dense, nslots, h_base,
                         c_begin, c_end);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// slice: state rows per CTA, 16, 32 or 64, or 0 for the library's choice.  A chunk step's MMA issue
// and hand-offs do not depend on the width and its epilogues scale with it: a 64-row step takes
// ~1.5x a 32-row one, a 16-row step ~0.75x.  So 64 rows when dv allows it and 1.5 x its waves of
// one CTA per SM are fewer than the 32-row grid's waves (many sequences or heads); 16 rows when
// twice the 32-row grid still fits one wave (few heads: the chain latency decides, and narrower
// slices shorten it); 32 otherwise.
template <int DK>
cudaError_t launch_chain_tc(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            const int32_t* cu, const int32_t* chunk_off, const int32_t* order, const void* ws,
                            const float* ws_rn, const float* init,
                            void* out, float* fin, int* err, int B, int T, int Hk, int Hv, int DV, int nc_dense,
                            long long nslots, int norm_qk, int h_base, int h_count, int c_begin, int c_end,
                            int slice, cudaStream_t st) {
  const long long ttot = cu != nullptr ? (long long)T : (long long)B * T;
  const cuuint64_t tt = (cuuint64_t)(ttot > 0 ? ttot : 1);
  CUtensorMap mk, mq, mw;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)DK, (cuuint64_t)Hk, tt};
    const cuuint64_t strides[2] = {(cuuint64_t)DK * 2, (cuuint64_t)Hk * DK * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    if (!make_map(&mk, k, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mq, q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const long long rows = nslots * Hv * 128;
    const cuuint64_t dims[2] = {64, (cuuint64_t)(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {64, 128};
    if (!make_map(&mw, ws, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  }
  if (slice == 0) {
    slice = 32;
    {
      int dev = 0, sms = 0;
      cudaError_t e;
      if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
      const long long n32 = (long long)B * (DV / 32) * h_count;
      const long long waves32 = (n32 + sms - 1) / sms, waves64 = (n32 / 2 + sms - 1) / sms;
      if (DV % 64 == 0 && 3 * waves64 < 2 * waves32) slice = 64;
      else if (2 * n32 <= sms) slice = 16;
    }
  }
  if (slice == 64) {
    if (DV % 64 != 0) return cudaErrorInvalidValue;
    return launch_chain_tc_dvt<DK, 64>(mk, mq, v, mw, g, beta, cu, chunk_off, order, ws_rn, init, out, fin, err, B,
                                       T, Hk, Hv, DV, nc_dense, nslots, norm_qk, h_base, h_count, c_begin, c_end,
                                       tt, st);
  }
  if (slice == 16)
    return launch_chain_tc_dvt<DK, 16>(mk, mq, v, mw, g, beta, cu, chunk_off, order, ws_rn, init, out, fin, err, B,
                                       T, Hk, Hv, DV, nc_dense, nslots, norm_qk, h_base, h_count, c_begin, c_end,
                                       tt, st);
  if (slice != 32) return cudaErrorInvalidValue;
  return launch_chain_tc_dvt<DK, 32>(mk, mq, v, mw, g, beta, cu, chunk_off, order, ws_rn, init, out, fin, err, B, T,
                                     Hk, Hv, DV, nc_dense, nslots, norm_qk, h_base, h_count, c_begin, c_end, tt, st);
}

#define GDN_INST_CHAIN_TC(DK)                                                                                \
  template cudaError_t launch_chain_tc<DK>(const void*, const void*, const void*, const float*, const float*, \
                                           const int32_t*, const int32_t*, const int32_t*, const void*,       \
                                           const float*, const float*, void*,                                 \
                                           float*, int*, int, int, int, int, int, int, long long, int, int,   \
                                           int, int, int, int, cudaStream_t);
GDN_INST_CHAIN_TC(32)
GDN_INST_CHAIN_TC(64)
GDN_INST_CHAIN_TC(128)

}  // namespace gdn

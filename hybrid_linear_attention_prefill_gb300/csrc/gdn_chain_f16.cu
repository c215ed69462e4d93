// Chunk-sequential state carry with fp16 tensor-core operands: the library's default.
//
// It runs the chunk recurrence of the wide-range state carry (gdn_chain_tc.cu), one CTA per
// (sequence, value head, 16-, 32- or 64-row slice of S), 8 epilogue warps and 1 issue warp,
// the slice of S in fp32 registers.  Per 64-token chunk, with Tm = (I + A)^-1 and PT = P Tm
// from the preparation kernel, gamma = cumsum(g), e = exp(gamma), d = exp(gamma_last - gamma):
//
//   phase 1   [X; Y] = [K; Q] S^T                       (M = 128 stacked tokens, K = dk)
//             R      = diag(beta) V - diag(beta e) X
//   phase 2   [U; Z] = [Tm; PT] R                       (M = 128, K = 64)
//             O      = scale (diag(e) Y + Z)            -> bf16 outputs
//   phase 3   dS^T   = K^T diag(d) U                    (M = dk = 128, K = 64)
//             S      = e_last S + dS
//
// the chunk form of S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T, o_t = S_t q_t / sqrt(dk)
// (the "chunked Gated DeltaNet prefill" of the "Open-Jev-27B-v1.1 native text worker" page,
// "Validation and optimization scope").
//
// Operands.  Every tensor-core operand is one fp16 value (kind::f16, fp32 accumulate): K and Q
// come from the preparation kernel as an fp16 image of the shared-memory tile, Tm and PT are
// fp16 there as well, and the state-side operands S, R and diag(d) U are rounded to fp16 from
// the fp32 values the epilogues hold.  fp16 keeps 11 significant bits where bf16 keeps 8, so a
// single fp16 operand replaces the bf16 hi + lo pair of the wide-range kernel: the MMAs carry
// N = DVT columns instead of 2 DVT, and the epilogues read and store half as many.  A float64
// model of the chunked path with these rounding points puts its errors below those of the bf16
// kernels (final state 4.6e-4 against 1.05e-3 relative, output 5.7e-4 against 2.5e-3 of the
// largest, on a no-decay, beta = 0.999 stress case): bf16 Tm was their largest rounding.
// fp16 stops at 65504.  An operand beyond it becomes infinite, and that reaches the state, so
// a (sequence, head) whose final fp32 state is not finite sets status bit 16 (also for
// non-finite inputs).  At the other end, fp16 keeps 11 bits only down to 2^-14; a state whose
// entries all stay below 2^-12 (values of order 1e-5 and less) has lost accuracy in its
// operands, so with check_small a CTA whose final state slice is nonzero but below 2^-12 sets
// status bit 32.  The wide-range kernel takes values of any magnitude.
//
// Shared-memory layouts (tile bases 1024-byte aligned):
//   [K; Q]   K-major, 128 B swizzle: [dk/64 blocks][128 rows][128 B]; rows 0..63 K, 64..127 Q
//            (the preparation kernel's image, one bulk copy per block).  The same K rows, read
//            MN-major (dk contiguous), are phase 3's A operand.
//   [Tm; PT] K-major, 128 B swizzle: [128 rows][128 B].
//   S, R, U  MN-major, 128 B swizzle: one 128-byte row per K index (d or token), whose first
//            DVT fp16 values are the slice's columns (N = DVT of the row's 64).
//   V        the bf16 value slice: 32 B rows unswizzled (16 rows), 64 B rows with the 64 B
//            swizzle (32), 128 B rows with the 128 B swizzle (64).
#include <cuda_fp16.h>

#include "gdn_tc.cuh"
#include "gdn_tmap.cuh"

namespace gdn {

namespace {

constexpr int kThreads = 288;  // 8 epilogue warps + 1 issue warp
constexpr int kEpiThreads = 256;
constexpr int kParts = 1;  // TMEM accumulators per phase (two in phase 1 measured 2 % slower)
constexpr uint32_t kMaxPolls = 1u << 24;
constexpr int kStatusNonFinite = 16;
constexpr int kStatusSmallState = 32;
constexpr float kSmallState = 1.f / 4096.f;  // 2^-12: two bits above fp16's smallest normal value

template <int DVT>
struct CfgH {
  static constexpr int kN = DVT;                       // MMA N: one fp16 column per state row
  static constexpr int kPS = kN < 32 ? 32 : kN;        // TMEM columns between phase 1's partials
  static constexpr uint32_t kTmemCols = kParts * kPS;  // 32, 32, 64
  static constexpr int kCPT = DVT / 2;                 // state columns per epilogue thread
  static constexpr int kGW = kCPT < 16 ? kCPT : 16;    // columns an epilogue step works on
  static constexpr int kNG = kCPT / kGW;               // steps per thread
  // stage layout (bytes)
  static constexpr int kOffKQ = 0;              // 2 x 16384
  static constexpr int kOffTP = 32768;          // 16384
  static constexpr int kOffV = kOffTP + 16384;  // 64 rows x 2 DVT bytes
  static constexpr int kVBytes = 64 * 2 * DVT;
  static constexpr int kOffG = kOffV + kVBytes;  // 64 fp32
  static constexpr int kOffB = kOffG + 256;      // 64 fp32
  static constexpr int kStage = (kOffB + 256 + 1023) / 1024 * 1024;  // 51, 53, 57 KB
  static constexpr int kStages = 3;  // chunk c + 2 loads during chunk c
  // B operands after the stages: S (128 d rows), R and dU (64 token rows), 128 B a row
  static constexpr int kOffS = kStages * kStage;
  static constexpr int kOffR = kOffS + 16384;
  static constexpr int kOffU = kOffR + 8192;
  // 64 rows: the Y rows of the output warps wait here between phases 1 and 2 ([32 columns][128 threads])
  static constexpr int kOffY = kOffU + 8192;
  static constexpr int kYBytes = DVT == 64 ? 32 * 128 * 4 : 0;
  static constexpr int kOffBar = kOffY + kYBytes;  // 3 MMA mbarriers, 3 load mbarriers, TMEM base, abort flag
  static constexpr int kSmemBytes = kOffBar + 64 + 1024;  // + slack for 1024-byte alignment
  static constexpr uint32_t kID_KS = tc::idesc_f16(128, kN, 0, 1);  // A K-major, B MN-major
  static constexpr uint32_t kID_KT = tc::idesc_f16(128, kN, 1, 1);  // A MN-major, B MN-major
  static_assert(DVT == 16 || DVT == 32 || DVT == 64, "16, 32 or 64 state rows per CTA");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert((3 + kStages) * 8 <= 48, "mbarriers in the barrier block");
};

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// W columns (8 or 16) of the warp's 32 TMEM lanes, summed over NP (1 or 2) accumulators PS
// columns apart.  The loads and their wait are one statement, so no use of the results can be
// scheduled before the wait.
template <int NP, int PS, int W>
__device__ __forceinline__ void tmem_sum(uint32_t taddr, float (&acc)[W]) {
  static_assert(NP == 1 || NP == 2, "one or two accumulators");
  if constexpr (W == 8 && NP == 1) {
    tc::tmem_ld8(taddr, acc);
  } else if constexpr (W == 16 && NP == 1) {
    tc::tmem_ld16(taddr, acc);
  } else if constexpr (W == 8) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr), "r"(taddr + PS)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = __uint_as_float(r[i]) + __uint_as_float(r[8 + i]);
  } else {
    static_assert(W == 16, "8 or 16 columns");
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr), "r"(taddr + PS)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = __uint_as_float(r[i]) + __uint_as_float(r[16 + i]);
  }
}

// W fp16 values at columns c0 .. c0 + W - 1 (c0 a multiple of 8) of operand row `row`:
// 16-byte chunks c0 / 8 .. of the 128-byte swizzled row.
template <int W>
__device__ __forceinline__ void store_h(unsigned char* tile, uint32_t row, int c0, const float* x) {
#pragma unroll
  for (int j = 0; j < W / 8; ++j)
    *reinterpret_cast<uint4*>(tile + tc::sw128(row, (uint32_t)(c0 / 8 + j))) =
        make_uint4(pack_h2(x[8 * j], x[8 * j + 1]), pack_h2(x[8 * j + 2], x[8 * j + 3]),
                   pack_h2(x[8 * j + 4], x[8 * j + 5]), pack_h2(x[8 * j + 6], x[8 * j + 7]));
}

// W bf16 values of token row `tok` of the value slice, columns c0 .. c0 + W - 1.
template <int DVT, int W>
__device__ __forceinline__ void load_v(const unsigned char* vt, int tok, int c0, float* vv) {
#pragma unroll
  for (int j = 0; j < W / 8; ++j) {
    const uint32_t ch = (uint32_t)(c0 / 8 + j);
    uint32_t off;
    if constexpr (DVT == 16) off = (uint32_t)tok * 32u + 16u * ch;
    else if constexpr (DVT == 32) off = tc::sw64((uint32_t)tok, ch);
    else off = tc::sw128((uint32_t)tok, ch);
    const uint4 raw = *reinterpret_cast<const uint4*>(vt + off);
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      vv[8 * j + 2 * p] = __uint_as_float(w4[p] << 16);
      vv[8 * j + 2 * p + 1] = __uint_as_float(w4[p] & 0xffff0000u);
    }
  }
}

}  // namespace

// One CTA per SM.  Nine warps leave three on one of the SM's four sub-partitions, whose 16 K
// registers then cap a thread at 168.
template <int DK, int DVT>
__global__ void __launch_bounds__(kThreads, 1)
gdn_chain_f16_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
                     const unsigned char* __restrict__ ws_kq, const float* __restrict__ g,
                     const float* __restrict__ beta, const int32_t* __restrict__ cu,
                     const int32_t* __restrict__ chunk_off, const int32_t* __restrict__ order, const float* init,
                     __nv_bfloat16* __restrict__ out, float* fin, int* __restrict__ err, int B, int T, int Hk,
                     int Hv, int DV, int nc_dense, long long nslots, int h_base, int c_begin, int c_end,
                     int check_small) {
  // The value tiles are inputs, ready before the preparation kernel finishes: for dense batches
  // the issue thread brings the first chunks' tiles into L2 before the wait below.
  if (cu == nullptr && threadIdx.x == 256) {
    const int nt = DV / DVT;
    const int bb = (int)blockIdx.x / nt, d0 = ((int)blockIdx.x - bb * nt) * DVT, hh = h_base + (int)blockIdx.y;
    tc::prefetch_tensormap(&tm_v);
    for (int cc = c_begin; cc < c_begin + CfgH<DVT>::kStages && cc * kChunk < T; ++cc)
      tc::tma_prefetch_l2_3d(&tm_v, d0, hh, (int)((long long)bb * T + (long long)cc * kChunk));
  }
  using C = CfgH<DVT>;
  if (threadIdx.x == 0) {  // the barriers need nothing from the kernel before
    extern __shared__ unsigned char smem_raw[];
    const uint32_t r = smem_u32(smem_raw);
    uint64_t* bb = reinterpret_cast<uint64_t*>(smem_raw + (((r + 1023u) & ~1023u) - r) + C::kOffBar);
    for (int i = 0; i < 3 + C::kStages; ++i) tc::mbar_init(&bb[i], 1);
    tc::fence_mbar_init();
  }
  // Launched as a programmatic dependent of the kernel before it in the stream (the preparation
  // kernel): the CTA starts while that kernel's last CTAs run and waits here until it has
  // completed and its writes are visible (otherwise this returns at once).
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t pad = ((raw_s + 1023u) & ~1023u) - raw_s;
  unsigned char* sm = smem_raw + pad;
  const uint32_t sb = raw_s + pad;  // shared-window address of sm

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);  // [0..2] MMA phases
  uint64_t* full = bars + 3;                                       // [0..kStages) stage loaded
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffBar + 48);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kOffBar + 52);
  int* state_max = reinterpret_cast<int*>(sm + C::kOffBar + 56);  // bits of the largest |S| (non-negative floats order as ints)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool issuer = warp == 8;
  const int q4 = warp & 3;           // TMEM lane quadrant (epilogue warps)
  const int half = (warp >> 2) & 1;  // state columns kCPT half .. kCPT half + kCPT - 1
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
  constexpr int kKBlocks = DK > 64 ? 2 : 1;                  // 64-wide d blocks per tile
  constexpr uint32_t kTxBytes = kKBlocks * 16384 + C::kVBytes + 16384;
  constexpr int kAhead = C::kStages - 1;  // chunks whose tiles are in flight ahead of the current one
  constexpr int kCPT = C::kCPT, kGW = C::kGW, kNG = C::kNG;

  const SeqChunk sq = seq_bounds(cu, b, T);
  const int slot0 = cu == nullptr ? b * nc_dense : chunk_off[b];
  int nchunks = (sq.len + kChunk - 1) / kChunk;
  if ((long long)slot0 + nchunks > nslots) nchunks = slot0 < nslots ? (int)(nslots - slot0) : 0;
  // this launch walks chunks c0 .. c1 - 1 of the sequence, from `init` (the state before
  // chunk c0) to `fin` (the state after chunk c1 - 1)
  const int c0 = c_begin < nchunks ? c_begin : nchunks;
  const int c1 = c_end < nchunks ? c_end : nchunks;

  // ---- set-up: TMEM, barriers, zero d-block 1 when dk <= 64 --------------------
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, C::kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    *abort_flag = 0;
    *state_max = 0;
    tc::fence_mbar_init();
  }
  if (issuer && lane == 0) {
    tc::prefetch_tensormap(&tm_v);
    tc::prefetch_tensormap(&tm_w);
  }
  if (kKBlocks == 1 && !issuer) {  // phase 3 reads all 128 rows of K^T: the rows d >= 64 stay zero
    for (int e = tid; e < C::kStages * 1024; e += kEpiThreads) {
      const int stg = e >> 10, w = e & 1023;
      *reinterpret_cast<uint4*>(sm + stg * C::kStage + C::kOffKQ + 16384 + w * 16) = make_uint4(0, 0, 0, 0);
    }
  }

  // ---- initial state: thread (row d, half) holds S[kCPT half + i][d] ----------------
  const int d = row;
  float s[kCPT];
  if (!issuer) {
    const size_t base = ((size_t)b * Hv + h) * DV + dv0 + kCPT * half;
#pragma unroll
    for (int i = 0; i < kCPT; ++i) s[i] = (init != nullptr && d < DK) ? init[(base + i) * DK + d] : 0.f;
#pragma unroll
    for (int gg = 0; gg < kNG; ++gg) store_h<kGW>(sm + C::kOffS, d, kCPT * half + kGW * gg, s + kGW * gg);
  }
  tc::fence_proxy_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tq = tmem + ((uint32_t)(32 * q4) << 16);  // this warp's lanes

  // bulk copies and TMA for the tiles of chunk c into stage stg (one thread); g and beta by cp.async.
  auto load_tiles = [&](int c, int stg) {
    unsigned char* st = sm + stg * C::kStage;
    const int t0 = (int)(sq.bos + (long long)c * kChunk);
    const unsigned char* kq = ws_kq + ((size_t)(slot0 + c) * Hk + hk) * kws_kq_bytes(DK);
    tc::mbar_arrive_expect_tx(&full[stg], kTxBytes);
#pragma unroll
    for (int db = 0; db < kKBlocks; ++db) tc::bulk_load(st + C::kOffKQ + db * 16384, kq + db * 16384, 16384, &full[stg]);
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
    }
  };

  if (c1 > c0) {
    if (issuer && lane == 0)
      for (int a = 0; a < kAhead && c0 + a < c1; ++a) load_tiles(c0 + a, a);
    load_scalars(c0, 0);
  }
  cp_async_commit();

  const int tok = 32 * (q4 & 1) + lane;  // this thread's token in phases 1-2
  // shared-memory descriptors of the operands at stage 0 / their buffers (the issuer's MMAs)
  const uint64_t dKQ0 = tc::sdesc(sb + C::kOffKQ, 16, 1024, tc::kSw128);     // [K; Q], K-major
  const uint64_t dKT0 = tc::sdesc(sb + C::kOffKQ, 16384, 1024, tc::kSw128);  // K^T, MN-major
  const uint64_t dTP0 = tc::sdesc(sb + C::kOffTP, 16, 1024, tc::kSw128);     // [Tm; PT], K-major
  const uint64_t dS = tc::sdesc(sb + C::kOffS, 16384, 1024, tc::kSw128);     // S, MN-major
  const uint64_t dR = tc::sdesc(sb + C::kOffR, 8192, 1024, tc::kSw128);      // R, MN-major
  const uint64_t dU = tc::sdesc(sb + C::kOffU, 8192, 1024, tc::kSw128);      // dU, MN-major
  bool aborted = false;
  int c = c0;
  for (; c < c1; ++c) {
    const int ci = c - c0;  // position in this launch: stage and barrier phases
    const int stg = ci % C::kStages;
    const uint32_t par = (uint32_t)(ci & 1);
    unsigned char* st = sm + stg * C::kStage;
    cp_async_wait<0>();
    // The stage's tiles: the thread that issued their copies waits for them, then the barrier
    // below publishes them to every thread (it makes the accesses that thread requested and saw
    // complete visible to all the CTA's threads).  The epilogue warps read the value slice after
    // that barrier without waiting themselves: 256 waits on a completed phase cost the chunk step
    // ~4 % at the headline size.
    if (issuer && lane == 0 && !tc::mbar_wait(&full[stg], (uint32_t)((ci / C::kStages) & 1), kMaxPolls)) {
      *abort_flag = 1;
      atomicOr(err, 2);
    }
    __syncthreads();
    // Every thread reads the abort flag right after each barrier, so all of them leave the loop
    // at the same barrier; the issuing thread acts on it after issuing that phase's MMAs (which
    // an abort makes harmless), so the read is off its path to the tensor core.
    const int ab_top = *abort_flag;

    if (issuer) {
      // Descriptors: this stage's bases plus each MMA's offset, added to the start-address field
      // (byte offset / 16; shared addresses stay below 2^18, so the 14-bit field does not carry).
      const uint64_t dKQ = dKQ0 + (uint64_t)((uint32_t)(stg * C::kStage) >> 4);
      const uint64_t dKT = dKT0 + (uint64_t)((uint32_t)(stg * C::kStage) >> 4);
      const uint64_t dTP = dTP0 + (uint64_t)((uint32_t)(stg * C::kStage) >> 4);
      // ---- phase 1: [X; Y] = [K; Q] S^T --------------------------------------------
      if (lane == 0) {
        tc::fence_after();
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks) {
          const uint64_t a = dKQ + (uint64_t)(((ks >> 2) * 16384 + (ks & 3) * 32) >> 4);
          const uint64_t bd = dS + (uint64_t)((ks * 2048) >> 4);
          tc::mma_bf16(tmem + C::kPS * (ks % kP1), a, bd, C::kID_KS, ks >= kP1);
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
      // ---- phase 2: [U; Z] = [Tm; PT] R ---------------------------------------------
      if (lane == 0) {
        tc::fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem, dTP + (uint64_t)((ks * 32) >> 4), dR + (uint64_t)((ks * 2048) >> 4), C::kID_KS, ks > 0);
        tc::commit(&bars[1]);
      }
      __syncwarp();
      if (ab_r) { aborted = true; break; }
      __syncthreads();  // dU written
      const int ab_d = *abort_flag;
      // ---- phase 3: dS^T = K^T dU ---------------------------------------------------
      if (lane == 0) {
        tc::fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem, dKT + (uint64_t)((ks * 2048) >> 4), dU + (uint64_t)((ks * 2048) >> 4), C::kID_KT, ks > 0);
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

    // ---- phase-1 epilogue: R = beta V - beta e X (rows 0..63), keep Y (rows 64..127)
    if (!tc::mbar_wait(&bars[0], par, kMaxPolls)) { *abort_flag = 1; atomicOr(err, 1); }
    tc::fence_after();
    // Y of the output warps (q4 >= 2) until phase 2: in registers (16, 32 rows), or in shared
    // memory (64 rows; column-major over the 128 output threads)
    float y[kNG][kGW];
    float* ys = reinterpret_cast<float*>(sm + C::kOffY) + (q4 >= 2 ? 32 * (q4 - 2) + lane + 64 * half : 0);
#pragma unroll
    for (int gg = 0; gg < kNG; ++gg) {
      const int cc = kCPT * half + kGW * gg;  // slice column of this step
      float acc[kGW];
      tmem_sum<kP1, C::kPS, kGW>(tq + cc, acc);
      if (q4 < 2) {
        float vv[kGW];
        load_v<DVT, kGW>(st + C::kOffV, tok, cc, vv);
        const float be = b_t * e_t;
#pragma unroll
        for (int i = 0; i < kGW; ++i) acc[i] = b_t * vv[i] - be * acc[i];
        store_h<kGW>(sm + C::kOffR, tok, cc, acc);
      } else if constexpr (DVT == 64) {
#pragma unroll
        for (int i = 0; i < kGW; ++i) ys[(kGW * gg + i) * 128] = acc[i];
      } else {
#pragma unroll
        for (int i = 0; i < kGW; ++i) y[gg][i] = acc[i];
      }
    }
    if (q4 < 2) tc::fence_proxy_async();  // R is read by the tensor core next
    tc::fence_before();
    __syncthreads();  // R written
    if (*abort_flag) { aborted = true; break; }

    // ---- phase-2 epilogue: dU (rows 0..63); outputs from Z (rows 64..127) ------------
    if (!tc::mbar_wait(&bars[1], par, kMaxPolls)) { *abort_flag = 1; atomicOr(err, 1); }
    tc::fence_after();
    const int n = min(kChunk, sq.len - c * kChunk);
    __nv_bfloat16* orow = out + ((size_t)(sq.bos + (long long)c * kChunk + tok) * Hv + h) * DV + dv0;
    uint32_t o2[kNG][kGW / 2];
#pragma unroll
    for (int gg = 0; gg < kNG; ++gg) {
      const int cc = kCPT * half + kGW * gg;
      float acc[kGW];
      tmem_sum<1, C::kPS, kGW>(tq + cc, acc);
      if (q4 < 2) {
#pragma unroll
        for (int i = 0; i < kGW; ++i) acc[i] *= d_t;
        store_h<kGW>(sm + C::kOffU, tok, cc, acc);
      } else {
        const float es = scale * e_t;
#pragma unroll
        for (int p = 0; p < kGW / 2; ++p) {
          float y0, y1;
          if constexpr (DVT == 64) { y0 = ys[(kGW * gg + 2 * p) * 128]; y1 = ys[(kGW * gg + 2 * p + 1) * 128]; }
          else { y0 = y[gg][2 * p]; y1 = y[gg][2 * p + 1]; }
          o2[gg][p] = pack_bf16(es * y0 + scale * acc[2 * p], es * y1 + scale * acc[2 * p + 1]);
        }
        if constexpr (DVT == 64) {  // stored now: the packed outputs do not stay live across the barrier
          if (tok < n) {
#pragma unroll
            for (int j = 0; j < kGW / 8; ++j)
              *reinterpret_cast<uint4*>(orow + cc + 8 * j) =
                  make_uint4(o2[gg][4 * j], o2[gg][4 * j + 1], o2[gg][4 * j + 2], o2[gg][4 * j + 3]);
          }
        }
      }
    }
    if (q4 < 2) tc::fence_proxy_async();  // dU is read by the tensor core next
    tc::fence_before();
    __syncthreads();  // dU written
    if (*abort_flag) { aborted = true; break; }

    // outputs go out while the phase-3 MMAs run
    if (DVT != 64 && q4 >= 2 && tok < n) {
#pragma unroll
      for (int gg = 0; gg < kNG; ++gg) {
        const int cc = kCPT * half + kGW * gg;
#pragma unroll
        for (int j = 0; j < kGW / 8; ++j)
          *reinterpret_cast<uint4*>(orow + cc + 8 * j) =
              make_uint4(o2[gg][4 * j], o2[gg][4 * j + 1], o2[gg][4 * j + 2], o2[gg][4 * j + 3]);
      }
    }

    // ---- phase-3 epilogue: S = e_last S + dS ------------------------------------------
    if (!tc::mbar_wait(&bars[2], par, kMaxPolls)) { *abort_flag = 1; atomicOr(err, 1); }
    tc::fence_after();
#pragma unroll
    for (int gg = 0; gg < kNG; ++gg) {
      const int cc = kCPT * half + kGW * gg;
      float acc[kGW];
      tmem_sum<1, C::kPS, kGW>(tq + cc, acc);
#pragma unroll
      for (int i = 0; i < kGW; ++i) s[kGW * gg + i] = fmaf(eC, s[kGW * gg + i], acc[i]);
      store_h<kGW>(sm + C::kOffS, d, cc, s + kGW * gg);
    }
    tc::fence_proxy_async();  // S is read by the tensor core at the next chunk
    tc::fence_before();
  }

  // ---- final state, clean-up -------------------------------------------------------
  cp_async_wait<0>();
  if (!aborted && !issuer && d < DK) {
    bool finite = true;
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < kCPT; ++i) {
      finite = finite && fabsf(s[i]) <= 3.402823466e38f;
      mx = fmaxf(mx, fabsf(s[i]));
    }
    if (!finite) atomicOr(err, kStatusNonFinite);
    if (check_small) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(__activemask(), mx, o));
      if (lane == 0) atomicMax(state_max, __float_as_int(mx));
    }
    if (fin != nullptr) {
      const size_t base = ((size_t)b * Hv + h) * DV + dv0 + kCPT * half;
#pragma unroll
      for (int i = 0; i < kCPT; ++i) fin[(base + i) * DK + d] = s[i];
    }
  }
  if (aborted && issuer && lane == 0) {
    // let MMAs and copies still in flight land before the CTA exits (bounded again)
    const int ci = c - c0;
    const uint32_t par = (uint32_t)(ci & 1);
    for (int i = 0; i < 3; ++i) (void)tc::mbar_wait(&bars[i], par, 1u << 16);
    for (int i = 0; i < C::kStages; ++i)
      (void)tc::mbar_wait(&full[(ci + i) % C::kStages], (uint32_t)(((ci + i) / C::kStages) & 1), 1u << 16);
  }
  tc::fence_before();
  __syncthreads();
  if (check_small && !aborted && tid == 0) {
    const float mx = __int_as_float(*state_max);
    if (mx > 0.f && mx < kSmallState) atomicOr(err, kStatusSmallState);
  }
  if (warp == 0) tc::tmem_dealloc(tmem, C::kTmemCols);
}

template <int DK, int DVT>
cudaError_t launch_chain_f16_dvt(const void* v, const CUtensorMap& mw, const void* ws_kq, const float* g,
                                 const float* beta, const int32_t* cu, const int32_t* chunk_off,
                                 const int32_t* order, const float* init, void* out, float* fin, int* err, int B,
                                 int T, int Hk, int Hv, int DV, int nc_dense, long long nslots, int h_base,
                                 int h_count, int c_begin, int c_end, int check_small, cuuint64_t tt,
                                 cudaStream_t st) {
  using C = CfgH<DVT>;
  CUtensorMap mv;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)DV, (cuuint64_t)Hv, tt};
    const cuuint64_t strides[2] = {(cuuint64_t)DV * 2, (cuuint64_t)Hv * DV * 2};
    const cuuint32_t box[3] = {DVT, 1, 64};
    const CUtensorMapSwizzle swz =
        DVT == 16 ? CU_TENSOR_MAP_SWIZZLE_NONE : DVT == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    if (!make_map16(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v, 3, dims, strides, box, swz))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = set_smem_limit_once<gdn_chain_f16_kernel<DK, DVT>>(C::kSmemBytes);
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
  e = cudaLaunchKernelEx(&cfg, gdn_chain_f16_kernel<DK, DVT>, mv, mw, static_cast<const unsigned char*>(ws_kq), g,
                         beta, cu, chunk_off, order, init, static_cast<__nv_bfloat16*>(out), fin, err, B, T, Hk,
                         Hv, DV, nc_dense, nslots, h_base, c_begin, c_end, check_small);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// check_small: report a final state below fp16's accurate range (status bit 32); off for the
// two-level scan's inner runs, whose transition states may be legitimately tiny.
// slice: state rows per CTA, 16, 32 or 64, or 0 for the library's choice.  The MMA issue and
// the hand-offs of a chunk step do not depend on the width and its epilogues scale with it:
// measured at 64 chunks, a 16-row step takes 0.91x a 32-row one and a 64-row step 1.41x.  So 64
// rows when dv allows it and 1.41 x its waves of one CTA per SM are fewer than the 32-row grid's
// waves (many sequences or heads); 16 rows when twice the 32-row grid still fits one wave (few
// heads: the chain latency decides, and narrower slices shorten it); 32 otherwise.
template <int DK>
cudaError_t launch_chain_f16(const void* v, const float* g, const float* beta, const int32_t* cu,
                             const int32_t* chunk_off, const int32_t* order, const void* ws, const void* ws_kq,
                             const float* init, void* out, float* fin, int* err, int B, int T, int Hk, int Hv,
                             int DV, int nc_dense, long long nslots, int h_base, int h_count, int c_begin,
                             int c_end, int slice, int check_small, cudaStream_t st) {
  const long long ttot = cu != nullptr ? (long long)T : (long long)B * T;
  const cuuint64_t tt = (cuuint64_t)(ttot > 0 ? ttot : 1);
  CUtensorMap mw;
  {
    const long long rows = nslots * Hv * 128;
    const cuuint64_t dims[2] = {64, (cuuint64_t)(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {64, 128};
    if (!make_map16(&mw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ws, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  if (slice == 0) {
    slice = 32;
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    const long long n32 = (long long)B * (DV / 32) * h_count;
    const long long waves32 = (n32 + sms - 1) / sms, waves64 = (n32 / 2 + sms - 1) / sms;
    if (DV % 64 == 0 && 141 * waves64 < 100 * waves32) slice = 64;
    else if (2 * n32 <= sms) slice = 16;
  }
  switch (slice) {
    case 16:
      return launch_chain_f16_dvt<DK, 16>(v, mw, ws_kq, g, beta, cu, chunk_off, order, init, out, fin, err, B, T, Hk,
                                          Hv, DV, nc_dense, nslots, h_base, h_count, c_begin, c_end, check_small,
                                          tt, st);
    case 32:
      return launch_chain_f16_dvt<DK, 32>(v, mw, ws_kq, g, beta, cu, chunk_off, order, init, out, fin, err, B, T, Hk,
                                          Hv, DV, nc_dense, nslots, h_base, h_count, c_begin, c_end, check_small,
                                          tt, st);
    case 64:
      if (DV % 64 != 0) return cudaErrorInvalidValue;
      return launch_chain_f16_dvt<DK, 64>(v, mw, ws_kq, g, beta, cu, chunk_off, order, init, out, fin, err, B, T, Hk,
                                          Hv, DV, nc_dense, nslots, h_base, h_count, c_begin, c_end, check_small,
                                          tt, st);
    default:
      return cudaErrorInvalidValue;
  }
}

#define GDN_INST_CHAIN_F16(DK)                                                                                 \
  template cudaError_t launch_chain_f16<DK>(const void*, const float*, const float*, const int32_t*,           \
                                            const int32_t*, const int32_t*, const void*, const void*,          \
                                            const float*, void*, float*, int*, int, int, int, int, int, int,   \
                                            long long, int, int, int, int, int, int, cudaStream_t);
GDN_INST_CHAIN_F16(32)
GDN_INST_CHAIN_F16(64)
GDN_INST_CHAIN_F16(128)

}  // namespace gdn

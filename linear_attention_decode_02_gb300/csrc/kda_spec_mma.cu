// Packed speculative decode (ragged cu_seqlens, T >= 1 tokens per row) in
// the chunked form on the 5th-generation tensor cores, bfloat16 state.
//
// For one (row, head) unit and a chunk of nt <= MT tokens starting from the
// state S (128 x 128, S[k][v]), with G_t the running sum of the log decays
// g_0 .. g_t (per key channel), P_t = exp(G_t), and q_t, k_t L2-normalised,
// the nt sequential delta-rule steps equal, with X_i = k_i / P_i,
// Y_t = P_t k_t and Z_t = P_t q_t:
//     a_t = S^T Y_t                  b_t = S^T Z_t
//     A_ti = X_i . Y_t (i < t)       B_ti = X_i . Z_t (i <= t)
//     u_t = beta_t (v_t - a_t - sum_{i<t} A_ti u_i)
//     o_t = scale (b_t + sum_{i<=t} B_ti u_i)
//     S'  = diag(P_end) (S + sum_i X_i u_i^T)
// (substitute S_{t-1} = diag(P_{t-1}) (S + sum_{i<t} X_i u_i^T) into the
// single step).  A chunk ends early once the summed largest per-token decay
// passes 80, and log decays are floored at -60, so P and 1/P stay finite in
// float32 (the same rule as the per-token kernel).  The two products with
// the state are dense contractions:
//   GEMM 1: S^T [Y | Z] : M = 128 value columns, N = 6 MT (each operand as
//           the sum of three bf16 pieces), K = 128 key rows; the state tile
//           is the A operand exactly as TMA loads it (MN-major);
//   GEMM 2: [X](128 x nt) [u](nt x 128): M = 128 key rows, N = 128, K = 48
//           holding the six piece products x_i u_j with i + j <= 4.
// A float32 value is the sum of three bf16 pieces to within 2^-24 of itself,
// so both products carry float32 accuracy.  GEMM 2 accumulates onto the
// state itself: the accumulator (float32, tensor memory) is first seeded with
// S by an MMA of the identity (held in tensor memory) and the TMA-loaded
// tile, so the epilogue only scales each key row by P_end and rounds to bf16
// once.  Rows longer than a chunk run chunk after chunk: between chunks the
// float32 state stays in the accumulator, and a bf16 high part (in the stage)
// plus a bf16 low part serve as the next GEMM 1's A operand.
//
// One persistent CTA per SM walks its units; warps are specialised:
//   warp 0      TMA loads of state blocks into a ring of MS stages;
//   warp 1      allocates tensor memory; one thread issues the MMAs;
//   warps 2-5   per chunk: token loads, L2 norms, cumulative decays, the
//               chunk length, the GEMM operands [Y | Z] and [X] (three bf16
//               pieces each), the pair sums A, B (reduce-scatter across the
//               warp), P_end;
//   warps 6-9   per chunk: read GEMM 1 from tensor memory (thread = value
//               column), forward substitution for u, outputs, u operand;
//               then read GEMM 2 (thread = key row), form S' in the stage
//               and store it with TMA.
// Operand buffers are double-buffered by chunk parity, so the prologue of
// the next chunk overlaps the epilogue of this one.  Every mbarrier wait is
// bounded in time: a role whose wait times out records a bit in the error
// word, raises the CTA's abort flag and leaves its loop; every role then
// meets at the final barrier before the tensor memory is freed.
#include <atomic>

#include "kda_stream_common.cuh"
#include "kda_tcgen05.cuh"

namespace kda {

// bit 3: a wait of the tensor-core speculative kernel timed out.
__device__ unsigned int g_kda_mma_error = 0;

namespace {

constexpr int MT = 8;                     // tokens per chunk
constexpr int MS = 3;                     // state stages
constexpr int NAB = MT * (MT - 1) / 2 + MT * (MT + 1) / 2;  // 28 A + 36 B pair sums
constexpr int NPRO = 8;                   // prologue warps, one token of the chunk each
constexpr int PRO_THREADS = NPRO * 32;
constexpr int EPI_WARP0 = 2 + NPRO;       // first epilogue warp
constexpr int MMA_THREADS = (EPI_WARP0 + 4) * 32;
constexpr float kMaxChunkDecay = 80.f;    // chunk bound on the summed largest per-token decay
constexpr float kLogDecayFloor = -60.f;
constexpr uint32_t TMEM_COLS = 512;       // D1 x 2 (64 columns), state accumulator x 2 (128), identity (64)
constexpr uint32_t D1_STRIDE = 64;
constexpr uint32_t ACC_COL = 128;         // accumulator of unit parity p: ACC_COL + 128 p
constexpr uint32_t IDENT_COL = 384;       // 128 x 128 bf16 identity (A operand), two per column
constexpr int N1 = 6 * MT;                // GEMM 1 columns: [Y | Z] x three pieces

constexpr uint32_t SZ_STATE = 32768;      // bf16 128 x 128
constexpr uint32_t SZ_W1A = N1 * 128;     // one 64-wide K atom of [N1 rows][128 k], K-major
constexpr uint32_t SZ_W1 = 2 * SZ_W1A;
constexpr uint32_t SZ_W2 = SZ_W1;         // [48 K rows][128 k], MN-major (A of GEMM 2): two 64-wide M atoms
constexpr uint32_t SZ_U2 = 16384;         // [128 rows][48 K], K-major, 128-byte rows
constexpr uint32_t O_STAGE = 0;
constexpr uint32_t O_LO = O_STAGE + MS * SZ_STATE;
constexpr uint32_t O_W1 = O_LO + SZ_STATE;
constexpr uint32_t O_W2 = O_W1 + 2 * SZ_W1;
constexpr uint32_t O_U2 = O_W2 + 2 * SZ_W2;
constexpr uint32_t O_KH = O_U2 + SZ_U2;             // float [MT][128] normalised keys
constexpr uint32_t O_QH = O_KH + MT * 128 * 4;      // float [MT][128] normalised queries
constexpr uint32_t O_G = O_QH + MT * 128 * 4;       // float [MT][128] floored log decays
constexpr uint32_t O_X = O_G + MT * 128 * 4;        // float [MT][128] X_i = k_i / P_i
constexpr uint32_t O_V = O_X + MT * 128 * 4;        // float [2][MT][128] values
constexpr uint32_t O_PEND = O_V + 2 * MT * 128 * 4; // float [2][128] P_end
constexpr uint32_t O_AB = O_PEND + 2 * 128 * 4;     // float [2][NAB] pair sums
constexpr uint32_t O_BETA = O_AB + 2 * NAB * 4;     // float [2][MT]
constexpr uint32_t O_GM = O_BETA + 2 * MT * 4;      // float [MT] largest decay of each staged token
constexpr uint32_t O_CHUNK = O_GM + MT * 4;         // int2 [2] (tokens, last) of the chunk in each buffer
constexpr uint32_t O_BAR = O_CHUNK + 2 * 8;
// full[MS] empty[MS] wready[2] efree[2] d1full[2] uready d2full sready pbar[2] ebar
constexpr int NBAR = 2 * MS + 12;
constexpr uint32_t O_MISC = O_BAR + NBAR * 8;       // TMEM base, abort flag
constexpr uint32_t O_END = O_MISC + 16;
constexpr size_t MMA_SMEM = O_END + 1024;           // + alignment slack of the base
static_assert(MMA_SMEM <= 232448, "stages exceed the 227 KB shared memory of a CTA");
static_assert(MT == 8 && NPRO == MT, "one prologue warp per token; its pair sums fill 16 reduce-scatter slots");
static_assert(SZ_W1A % 1024 == 0 && N1 % 16 == 0, "GEMM 1 operand atoms and N");
static_assert(O_LO % 1024 == 0 && O_W1 % 1024 == 0 && O_W2 % 1024 == 0 && O_U2 % 1024 == 0,
              "operand atoms must be 1024-byte aligned");

// GEMM 1: M = 128 (A = state, MN-major), N = N1 (B K-major); GEMM 2: M = N = 128 (A MN-major, B K-major).
constexpr uint32_t ID1 = tc::idesc_bf16(128, N1, true, false);
constexpr uint32_t ID2 = tc::idesc_bf16(128, 128, true, false);
// Seeding the accumulator with the state: I (A, in tensor memory) times S (B, MN-major).
constexpr uint32_t IDS = tc::idesc_bf16(128, 128, false, true);

__device__ __forceinline__ void record_mma_error() { atomicOr(&g_kda_mma_error, 8u); }

// Waits for the phase of `bar` with the given parity.  Each try may suspend
// the thread for up to 0.2 ms (it wakes as soon as the phase completes), so
// waiting warps take no issue slots from the working ones; false after
// kWaitNs in total.
__device__ __forceinline__ bool mbar_sleep_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (true) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(200000u)
        : "memory");
    if (done) return true;
    if (global_ns() - t0 > kWaitNs) return false;
  }
}

// Shared -> global TMA tensor store (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_addr(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}

// Byte offset of element (row, k) of a K-major operand with 128 K per row
// held as two 64-wide K atoms of N1 x 128 B each.
__device__ __forceinline__ uint32_t w1_offset(int row, int k) {
  return (uint32_t)(k >> 6) * SZ_W1A + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) + (k & 7) * 2;
}
// Byte offset of 16-byte chunk c of row r of a K-major operand with 128-byte rows.
__device__ __forceinline__ uint32_t row_chunk(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }


// Two floats as three bf16x2 pieces (low half = a): a = a1 + a2 + a3 to
// within 2^-24 |a| (bf16 keeps the float32 exponent range), likewise b.
__device__ __forceinline__ void split2x3(float a, float b, uint32_t& p1, uint32_t& p2, uint32_t& p3) {
  p1 = pack_bf2(a, b);
  const float ra = a - bf_lo(p1), rb = b - bf_hi(p1);
  p2 = pack_bf2(ra, rb);
  p3 = pack_bf2(ra - bf_lo(p2), rb - bf_hi(p2));
}

__device__ __forceinline__ float4 add4(float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }
__device__ __forceinline__ float4 mul4(float4 a, float4 b) { return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w); }
__device__ __forceinline__ float dot4(float4 a, float4 b) { return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w; }
__device__ __forceinline__ float4 exp4(float4 x) { return make_float4(expf(x.x), expf(x.y), expf(x.z), expf(x.w)); }

// Four floats as three 8-byte vectors of bf16 pieces (piece 1, 2, 3).
__device__ __forceinline__ void split4x3(float4 x, uint2 (&p)[3]) {
  uint32_t a0, b0, c0, a1, b1, c1;
  split2x3(x.x, x.y, a0, b0, c0);
  split2x3(x.z, x.w, a1, b1, c1);
  p[0] = make_uint2(a0, a1);
  p[1] = make_uint2(b0, b1);
  p[2] = make_uint2(c0, c1);
}

// Eight floats as three 16-byte vectors of bf16 pieces.
__device__ __forceinline__ void split8x3(const float (&x)[8], uint4& a, uint4& b, uint4& c) {
  uint32_t pa[4], pb[4], pc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) split2x3(x[2 * i], x[2 * i + 1], pa[i], pb[i], pc[i]);
  a = make_uint4(pa[0], pa[1], pa[2], pa[3]);
  b = make_uint4(pb[0], pb[1], pb[2], pb[3]);
  c = make_uint4(pc[0], pc[1], pc[2], pc[3]);
}

// Eight floats as bf16 high parts and the bf16 rounding of the remainders.
__device__ __forceinline__ void split8(const float (&x)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = pack_bf2(x[2 * i], x[2 * i + 1]);
    l[i] = pack_bf2(x[2 * i] - bf_lo(h[i]), x[2 * i + 1] - bf_hi(h[i]));
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Row bounds and slot of the units blockIdx.x + (j0 + lane) * gridDim.x,
// one unit per lane: (t0, t1, slot); t1 <= t0 for empty rows.
__device__ __forceinline__ int3 unit_meta(const SpecArgs& a, int j0, int n_my, int lane) {
  int3 m = make_int3(0, 0, 0);
  if (j0 + lane < n_my) {
    const int u = blockIdx.x + (j0 + lane) * gridDim.x;
    const int n = u / a.H;
    m.x = max(__ldg(a.cu + n), 0);
    m.y = min(__ldg(a.cu + n + 1), a.R);
    m.z = __ldg(a.idx + n);
  }
  return m;
}

}  // namespace

template <bool VERIFY>
__global__ void __launch_bounds__(MMA_THREADS, 1) kda_spec_mma_kernel(const SpecArgs a,
                                                                      const __grid_constant__ CUtensorMap map) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + O_BAR);
  uint64_t* empty = full + MS;
  uint64_t* wready = empty + MS;
  uint64_t* efree = wready + 2;
  uint64_t* d1full = efree + 2;
  uint64_t* uready = d1full + 2;
  uint64_t* d2full = uready + 1;
  uint64_t* sready = d2full + 1;
  uint64_t* pbar = sready + 1;  // prologue group barriers (2 per chunk)
  uint64_t* ebar = pbar + 2;    // epilogue group barrier before a state store
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(sm + O_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + O_MISC + 4);
  float* s_kh = reinterpret_cast<float*>(sm + O_KH);
  float* s_qh = reinterpret_cast<float*>(sm + O_QH);
  float* s_g = reinterpret_cast<float*>(sm + O_G);
  float* s_x = reinterpret_cast<float*>(sm + O_X);
  float* s_gm = reinterpret_cast<float*>(sm + O_GM);
  int2* s_chunk = reinterpret_cast<int2*>(sm + O_CHUNK);
  float* s_v = reinterpret_cast<float*>(sm + O_V);
  float* s_pend = reinterpret_cast<float*>(sm + O_PEND);
  float* s_ab = reinterpret_cast<float*>(sm + O_AB);
  float* s_beta = reinterpret_cast<float*>(sm + O_BETA);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < MS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&wready[b], PRO_THREADS);
      mbar_init(&efree[b], 128);
      mbar_init(&d1full[b], 1);
    }
    mbar_init(uready, 128);
    mbar_init(d2full, 1);
    mbar_init(sready, 128);
    mbar_init(&pbar[0], PRO_THREADS);
    mbar_init(&pbar[1], PRO_THREADS);
    mbar_init(ebar, 128);
    *s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) tc::alloc(s_taddr, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = *s_taddr;
  if (warp >= EPI_WARP0) {  // the identity, once: lane k holds 1.0 (bf16 0x3F80) at K index k
    const int r = 32 * (warp & 3) + lane;
    const uint32_t one = (r & 1) ? 0x3F800000u : 0x00003F80u;
#pragma unroll
    for (int h32 = 0; h32 < 2; ++h32) {
      float z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = __uint_as_float(32 * h32 + i == (r >> 1) ? one : 0u);
      tc::st32(taddr + ((uint32_t)(32 * (warp & 3)) << 16) + IDENT_COL + 32 * h32, z);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  pdl_wait();
  pdl_launch_dependents();

  const int G = gridDim.x;
  const int n_my = (a.N * a.H - (int)blockIdx.x + G - 1) / G;  // units blockIdx.x + j * G
  const int64_t orow = (int64_t)a.H * kD;                       // output row stride
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  // Waits on `bar` for `parity`, warp-uniformly; on a timeout raises the abort flag.
  auto wait_or_abort = [&](uint64_t* bar, uint32_t parity) -> bool {
    const bool ok = mbar_sleep_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if (lane == 0) {
      record_mma_error();
      *s_abort = 1;
    }
    return false;
  };
  // Barrier of a 128-thread role group built on an mbarrier, so that it is
  // bounded in time like every other wait.
  auto group_sync = [&](uint64_t* bar, uint32_t parity) -> bool {
    mbar_arrive(bar);
    return wait_or_abort(bar, parity);
  };

  if (warp == 0) {
    // ---------------- producer: state blocks into the stage ring ----------------
    int L = 0;
    bool run = true;
    for (int j0 = 0; j0 < n_my && run; j0 += 32) {
      const int3 m = unit_meta(a, j0, n_my, lane);
      const int cnt = min(32, n_my - j0);
      for (int t = 0; t < cnt && run; ++t) {
        const int t0 = __shfl_sync(0xffffffffu, m.x, t), t1 = __shfl_sync(0xffffffffu, m.y, t);
        const int slot = __shfl_sync(0xffffffffu, m.z, t);
        if (t1 <= t0 || slot <= 0 || slot >= a.num_slots) continue;
        const int h = (blockIdx.x + (j0 + t) * G) % a.H;
        const int s = L % MS, round = L / MS;
        if (*s_abort || (round > 0 && !wait_or_abort(&empty[s], (round - 1) & 1))) { run = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], SZ_STATE);
          tma_load_state<__nv_bfloat16>(sm + O_STAGE + s * SZ_STATE, &map, h, slot, &full[s]);
        }
        {  // the unit's token rows into L2 (128-byte lines of q, k, v and g), ahead of the prologue
          const int qsz = a.qkv_dtype == KDA_DT_F32 ? 4 : 2;  // lines per 128-element row
          const int per = 3 * qsz + 4;
          const int ntok = min(t1 - t0, 32);
          for (int i = lane; i < ntok * per; i += 32) {
            const int64_t tk = t0 + i / per;
            const int p = i % per;
            const char* line;
            if (p < 3 * qsz) {
              const int which = p / qsz;
              const void* base = which == 0 ? a.q : (which == 1 ? a.k : a.v);
              const int64_t rs = which == 0 ? a.q_rs : (which == 1 ? a.k_rs : a.v_rs);
              const int64_t hs = which == 0 ? a.q_hs : (which == 1 ? a.k_hs : a.v_hs);
              line = static_cast<const char*>(base) + (tk * rs + (int64_t)h * hs) * qsz + (p % qsz) * 128;
            } else {
              line = reinterpret_cast<const char*>(a.g + tk * a.g_rs + (int64_t)h * a.g_hs) + (p - 3 * qsz) * 128;
            }
            asm volatile("prefetch.global.L2 [%0];" ::"l"(line));
          }
        }
        __syncwarp();
        ++L;
      }
    }
    // no load may still be writing shared memory when the CTA exits
    for (int s = 0; s < MS && s < L; ++s) {
      const int last = s + MS * ((L - 1 - s) / MS);
      mbar_sleep_wait(&full[s], (last / MS) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    int L = 0, it = 0, g2 = 0, nf = 0;
    uint64_t* last_bar = nullptr;
    uint32_t last_par = 0;
    bool run = true;
    for (int j0 = 0; j0 < n_my && run; j0 += 32) {
      const int3 m = unit_meta(a, j0, n_my, lane);
      const int cnt = min(32, n_my - j0);
      for (int t = 0; t < cnt && run; ++t) {
        const int t0 = __shfl_sync(0xffffffffu, m.x, t), t1 = __shfl_sync(0xffffffffu, m.y, t);
        const int slot = __shfl_sync(0xffffffffu, m.z, t);
        if (t1 <= t0 || slot <= 0 || slot >= a.num_slots) continue;
        const int s = L % MS;
        for (int c = 0;; ++c) {  // chunks: the prologue publishes each chunk's length and whether it is the last
          const int b = it & 1;
          const uint32_t bph = (it >> 1) & 1;
          bool ok = !*s_abort;
          if (ok) ok = c == 0 ? wait_or_abort(&full[s], (L / MS) & 1) : wait_or_abort(sready, (nf++) & 1);
          if (ok) ok = wait_or_abort(&wready[b], bph);
          if (!ok) { run = false; break; }
          const bool last = s_chunk[b].y != 0;
          if (lane == 0) {
            tc::fence_after_sync();
            const uint32_t st = smem_addr(sm + O_STAGE + s * SZ_STATE), lo = smem_addr(sm + O_LO);
            const uint32_t w1 = smem_addr(sm + O_W1 + b * SZ_W1);
            const uint32_t d1 = taddr + b * D1_STRIDE;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              tc::mma_bf16(d1, tc::desc_sw128(st + ks * 2048, 16384, 1024),
                           tc::desc_sw128(w1 + (ks >> 2) * SZ_W1A + (ks & 3) * 32, 16, 1024), ID1, ks > 0);
            if (c > 0) {  // carried state: add its low part
#pragma unroll
              for (int ks = 0; ks < 8; ++ks)
                tc::mma_bf16(d1, tc::desc_sw128(lo + ks * 2048, 16384, 1024),
                             tc::desc_sw128(w1 + (ks >> 2) * SZ_W1A + (ks & 3) * 32, 16, 1024), ID1, true);
            } else if (!VERIFY || !last) {  // the unit's accumulator starts as S (exactly, in float32)
#pragma unroll
              for (int ks = 0; ks < 8; ++ks)
                tc::mma_bf16_ta(taddr + ACC_COL + 128 * (L & 1), taddr + IDENT_COL + 8 * ks,
                                tc::desc_sw128(st + ks * 2048, 16384, 1024), IDS, ks > 0);
            }
            tc::commit(&d1full[b]);
          }
          __syncwarp();
          last_bar = &d1full[b];
          last_par = bph;
          if (!VERIFY || !last) {
            if (!wait_or_abort(uready, g2 & 1)) { run = false; break; }
            if (lane == 0) {
              tc::fence_after_sync();
              const uint32_t w2 = smem_addr(sm + O_W2 + b * SZ_W2), u2 = smem_addr(sm + O_U2);
#pragma unroll
              for (int ks = 0; ks < 3; ++ks)  // accumulator += X u^T
                tc::mma_bf16(taddr + ACC_COL + 128 * (L & 1), tc::desc_sw128(w2 + ks * 2048, SZ_W1A, 1024),
                             tc::desc_sw128(u2 + ks * 32, 16, 1024), ID2, true);
              tc::commit(d2full);
            }
            __syncwarp();
            last_bar = d2full;
            last_par = g2 & 1;
            ++g2;
          }
          ++it;
          if (last) break;
        }
        ++L;
      }
    }
    // every MMA this thread issued has completed before the columns are freed
    if (last_bar != nullptr) mbar_sleep_wait(last_bar, last_par);
  } else if (warp < EPI_WARP0) {
    // ---------------- prologue: operands of each chunk ----------------
    const int pw = warp - 2;
    const int ptid = threadIdx.x - 64;  // 0 .. PRO_THREADS - 1
    // padding token rows outside [cu[0], cu[N]): zero output, shared by all CTAs
    {
      const int lo = min(max(__ldg(a.cu), 0), a.R);
      const int hi = max(min(__ldg(a.cu + a.N), a.R), lo);
      const int64_t per_row = (int64_t)a.H * 16;  // 16-byte pieces of one output row
      const int64_t total = ((int64_t)lo + (a.R - hi)) * per_row;
      for (int64_t i = (int64_t)blockIdx.x * PRO_THREADS + ptid; i < total; i += (int64_t)G * PRO_THREADS) {
        const int64_t rr = i / per_row;
        const int64_t row = rr < lo ? rr : hi + (rr - lo);
        *reinterpret_cast<uint4*>(out + row * orow + (i % per_row) * 8) = make_uint4(0, 0, 0, 0);
      }
    }
    int it = 0;
    bool run = true;
    for (int j0 = 0; j0 < n_my && run; j0 += 32) {
      const int3 m = unit_meta(a, j0, n_my, lane);
      const int cnt = min(32, n_my - j0);
      for (int t = 0; t < cnt && run; ++t) {
        const int t0 = __shfl_sync(0xffffffffu, m.x, t), t1 = __shfl_sync(0xffffffffu, m.y, t);
        const int slot = __shfl_sync(0xffffffffu, m.z, t);
        if (t1 <= t0) continue;
        const int h = (blockIdx.x + (j0 + t) * G) % a.H;
        if (slot <= 0 || slot >= a.num_slots) {  // null row: zero its token rows, touch no cache
          for (int i = ptid; i < (t1 - t0) * 16; i += PRO_THREADS)
            *reinterpret_cast<uint4*>(out + (int64_t)(t0 + i / 16) * orow + h * kD + (i % 16) * 8) =
                make_uint4(0, 0, 0, 0);
          continue;
        }
        for (int tok0 = t0; tok0 < t1; ++it) {
          const int b = it & 1;
          if (*s_abort || (it >= 2 && !wait_or_abort(&efree[b], ((it >> 1) - 1) & 1))) { run = false; break; }
          const int nl = min(MT, t1 - tok0);  // tokens staged; the chunk may take fewer
          const int c4 = 4 * lane;
          // 1. one warp per token j = pw: load, normalise, floor the log decays, stage
          const int j = pw;
          if (j < nl) {
            const int64_t tk = tok0 + j;
            const float4 qj = load4(a.q, tk * a.q_rs + (int64_t)h * a.q_hs + c4, a.qkv_dtype);
            const float4 kj = load4(a.k, tk * a.k_rs + (int64_t)h * a.k_hs + c4, a.qkv_dtype);
            const float4 vj = load4(a.v, tk * a.v_rs + (int64_t)h * a.v_hs + c4, a.qkv_dtype);
            const float4 graw = __ldg(reinterpret_cast<const float4*>(a.g + tk * a.g_rs + (int64_t)h * a.g_hs + c4));
            const float braw = lane == 0 ? load1(a.beta, tk * a.b_rs + (int64_t)h * a.b_hs, a.beta_dtype) : 0.f;
            if (VERIFY && a.kg != nullptr && tok0 - t0 + j < a.t_cap) {
              float* kgp = a.kg + (((int64_t)slot * a.H + h) * a.t_cap + tok0 - t0 + j) * (2 * kD);
              reinterpret_cast<float4*>(kgp)[lane] = kj;
              reinterpret_cast<float4*>(kgp + kD)[lane] = graw;
            }
            const float4 gj = make_float4(fmaxf(graw.x, kLogDecayFloor), fmaxf(graw.y, kLogDecayFloor),
                                          fmaxf(graw.z, kLogDecayFloor), fmaxf(graw.w, kLogDecayFloor));
            float qq = qj.x * qj.x + qj.y * qj.y + qj.z * qj.z + qj.w * qj.w;
            float kk = kj.x * kj.x + kj.y * kj.y + kj.z * kj.z + kj.w * kj.w;
            float gm = fmaxf(fmaxf(-gj.x, -gj.y), fmaxf(-gj.z, -gj.w));
            qq = warp_sum(qq);
            kk = warp_sum(kk);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
            const float rq = rsqrtf(qq + kL2Eps), rk = rsqrtf(kk + kL2Eps);
            reinterpret_cast<float4*>(s_kh + j * kD)[lane] = make_float4(kj.x * rk, kj.y * rk, kj.z * rk, kj.w * rk);
            reinterpret_cast<float4*>(s_qh + j * kD)[lane] = make_float4(qj.x * rq, qj.y * rq, qj.z * rq, qj.w * rq);
            reinterpret_cast<float4*>(s_g + j * kD)[lane] = gj;
            reinterpret_cast<float4*>(s_v + (b * MT + j) * kD)[lane] = vj;
            if (lane == 0) {
              s_beta[b * MT + j] = a.beta_is_logit ? sigmoidf_(braw) : braw;
              s_gm[j] = gm;
            }
          }
          if (!group_sync(&pbar[0], it & 1)) { run = false; break; }
          // the chunk: the longest prefix whose summed largest decay stays within the bound
          int nt = 1;
          {
            float acc = s_gm[0];
            for (int j = 1; j < nl; ++j) {
              acc += s_gm[j];
              if (acc > kMaxChunkDecay) break;
              nt = j + 1;
            }
          }
          const bool last = tok0 + nt >= t1;
          if (ptid == 0) s_chunk[b] = make_int2(nt, last ? 1 : 0);
          // 2. token j = pw, lane = key rows 4 lane .. 4 lane + 3: its rows of
          // both GEMM operands ([Y | Z] and [X], three pieces each)
          unsigned char* w1 = sm + O_W1 + b * SZ_W1;
          unsigned char* w2 = sm + O_W2 + b * SZ_W2;
          const uint32_t o0 = w1_offset(j, c4);  // rows j + p MT (p = 0..5) share one swizzle phase
          float4 Y, Z;
          if (j >= nt) {  // K rows of absent tokens must be zero: they meet zero u rows in GEMM 2
#pragma unroll
            for (int p = 0; p < 6; ++p) *reinterpret_cast<uint2*>(w2 + o0 + p * MT * 128) = make_uint2(0u, 0u);
          } else {
            float4 Gj = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int i = 0; i <= j; ++i) Gj = add4(Gj, *reinterpret_cast<const float4*>(s_g + i * kD + c4));
            const float4 P = exp4(Gj);
            // 1 / P correctly rounded: P_i X_i = k_i to within an ulp
            const float4 R = make_float4(__frcp_rn(P.x), __frcp_rn(P.y), __frcp_rn(P.z), __frcp_rn(P.w));
            const float4 kj = *reinterpret_cast<const float4*>(s_kh + j * kD + c4);
            Y = mul4(P, kj);
            Z = mul4(P, *reinterpret_cast<const float4*>(s_qh + j * kD + c4));
            const float4 X = mul4(R, kj);
            reinterpret_cast<float4*>(s_x + j * kD)[lane] = X;
            if (j == nt - 1) reinterpret_cast<float4*>(s_pend + b * kD)[lane] = P;
            uint2 y[3], z[3], x[3];
            split4x3(Y, y);
            split4x3(Z, z);
            split4x3(X, x);
#pragma unroll
            for (int p = 0; p < 3; ++p) {  // GEMM 1 rows: [Y | Z] per piece
              *reinterpret_cast<uint2*>(w1 + o0 + (2 * p) * MT * 128) = y[p];
              *reinterpret_cast<uint2*>(w1 + o0 + (2 * p + 1) * MT * 128) = z[p];
            }
            // GEMM 2 K rows: x1 x1 x1 x2 x2 x3, against u1 u2 u3 u1 u2 u1
            *reinterpret_cast<uint2*>(w2 + o0) = x[0];
            *reinterpret_cast<uint2*>(w2 + o0 + MT * 128) = x[0];
            *reinterpret_cast<uint2*>(w2 + o0 + 2 * MT * 128) = x[0];
            *reinterpret_cast<uint2*>(w2 + o0 + 3 * MT * 128) = x[1];
            *reinterpret_cast<uint2*>(w2 + o0 + 4 * MT * 128) = x[1];
            *reinterpret_cast<uint2*>(w2 + o0 + 5 * MT * 128) = x[2];
          }
          if (!group_sync(&pbar[1], it & 1)) { run = false; break; }
          // 3. pair sums of token t = j: slots 0..7 = A_ti = X_i . Y_t (i < t),
          // 8..15 = B_ti = X_i . Z_t (i <= t), reduce-scattered over the warp
          if (j < nt) {
            float v[16];
#pragma unroll
            for (int i = 0; i < MT; ++i) {
              v[i] = 0.f;
              v[MT + i] = 0.f;
              if (i <= j) {
                const float4 xi = *reinterpret_cast<const float4*>(s_x + i * kD + c4);
                if (i < j) v[i] = dot4(xi, Y);
                v[MT + i] = dot4(xi, Z);
              }
            }
#pragma unroll
            for (int l = 0; l < 4; ++l) {  // lane l ends with slot l % 16 of its half-warp
              const int half = 8 >> l;
              const int bit = 3 - l;
              const bool up = (lane >> bit) & 1;
#pragma unroll
              for (int i = 0; i < half; ++i) {
                const float send = up ? v[i] : v[i + half];
                const float keep = up ? v[i + half] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1 << bit);
              }
            }
            const float tot = v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
            if (lane < j) s_ab[b * NAB + j * (j - 1) / 2 + lane] = tot;
            if (lane >= MT && lane <= MT + j) s_ab[b * NAB + MT * (MT - 1) / 2 + j * (j + 1) / 2 + lane - MT] = tot;
          }
          fence_proxy_async_smem();  // operands written here are read by the tensor cores
          mbar_arrive(&wready[b]);
          tok0 += nt;
        }
      }
    }
  } else {
    // ---------------- epilogue: substitution, outputs, state ----------------
    const int etid = threadIdx.x - EPI_WARP0 * 32;
    const int r = 32 * (warp & 3) + lane;  // this thread's tensor-memory lane
    const uint32_t tl = taddr + ((uint32_t)(32 * (warp & 3)) << 16);
    const bool elected = etid == 0;
    int L = 0, it = 0, g2 = 0, nstore = 0;
    int pend = -1;  // stage whose TMA store may still be reading shared memory
    bool run = true;
    for (int j0 = 0; j0 < n_my && run; j0 += 32) {
      const int3 m = unit_meta(a, j0, n_my, lane);
      const int cnt = min(32, n_my - j0);
      for (int t = 0; t < cnt && run; ++t) {
        const int t0 = __shfl_sync(0xffffffffu, m.x, t), t1 = __shfl_sync(0xffffffffu, m.y, t);
        const int slot = __shfl_sync(0xffffffffu, m.z, t);
        if (t1 <= t0 || slot <= 0 || slot >= a.num_slots) continue;
        const int h = (blockIdx.x + (j0 + t) * G) % a.H;
        const int s = L % MS;
        if (*s_abort || !wait_or_abort(&full[s], (L / MS) & 1)) { run = false; break; }
        unsigned char* st = sm + O_STAGE + s * SZ_STATE;
        for (int c = 0, tok0 = t0;; ++c) {  // chunks as the prologue published them
          const int b = it & 1;
          const uint32_t bph = (it >> 1) & 1;
          if (!wait_or_abort(&wready[b], bph) || !wait_or_abort(&d1full[b], bph)) { run = false; break; }
          const int2 ch = s_chunk[b];
          const int nt = ch.x;
          const bool last = ch.y != 0;
          tc::fence_after_sync();
          // ---- substitution: this thread is value column v = r
          float d1[64];  // columns N1 .. 63 are not written by GEMM 1 and not used
          tc::ld64(tl + b * D1_STRIDE, d1);
          float u[MT];
          const float* sv = s_v + b * MT * kD;
          const float* ab = s_ab + b * NAB;
#pragma unroll
          for (int j = 0; j < MT; ++j) {
            u[j] = 0.f;
            if (j < nt) {
              float acc = sv[j * kD + r] - (d1[j] + d1[2 * MT + j] + d1[4 * MT + j]);
#pragma unroll
              for (int i = 0; i < j; ++i) acc = fmaf(-ab[j * (j - 1) / 2 + i], u[i], acc);
              u[j] = s_beta[b * MT + j] * acc;
              float o = d1[MT + j] + d1[3 * MT + j] + d1[5 * MT + j];
#pragma unroll
              for (int i = 0; i <= j; ++i) o = fmaf(ab[MT * (MT - 1) / 2 + j * (j + 1) / 2 + i], u[i], o);
              out[(int64_t)(tok0 + j) * orow + h * kD + r] = __float2bfloat16_rn(a.scale * o);
              if (VERIFY && a.corr != nullptr && tok0 - t0 + j < a.t_cap)
                a.corr[(((int64_t)slot * a.H + h) * a.t_cap + tok0 - t0 + j) * kD + r] = u[j];
            }
          }
          const bool gemm2 = !VERIFY || !last;
          if (gemm2) {  // row v of the u operand, pieces u1..u3: K = [u1 | u2 | u3 | u1 | u2 | u1]
            uint4 u1, u2p, u3;
            split8x3(u, u1, u2p, u3);
            unsigned char* u2 = sm + O_U2;
            *reinterpret_cast<uint4*>(u2 + row_chunk(r, 0)) = u1;
            *reinterpret_cast<uint4*>(u2 + row_chunk(r, 1)) = u2p;
            *reinterpret_cast<uint4*>(u2 + row_chunk(r, 2)) = u3;
            *reinterpret_cast<uint4*>(u2 + row_chunk(r, 3)) = u1;
            *reinterpret_cast<uint4*>(u2 + row_chunk(r, 4)) = u2p;
            *reinterpret_cast<uint4*>(u2 + row_chunk(r, 5)) = u1;
            fence_proxy_async_smem();
          }
          tc::fence_before_sync();
          if (gemm2) mbar_arrive(uready);
          if (elected && pend >= 0) {  // the previous unit's store has read its stage: release it
            bulk_wait_read();
            mbar_arrive(&empty[pend]);
            pend = -1;
          }
          if (VERIFY && last && elected) mbar_arrive(&empty[s]);  // its last GEMM 1 has completed
          if (gemm2) {
            if (!wait_or_abort(d2full, g2 & 1)) { run = false; break; }
            ++g2;
            tc::fence_after_sync();
            // ---- S' = P_end (S + X u^T), the accumulator scaled per key row: this thread is row k = r
            const float2 P2 = dup2(s_pend[b * kD + r]);
            unsigned char* lo = sm + O_LO;
            const uint32_t acc = tl + ACC_COL + 128 * (L & 1);
#pragma unroll 1
            for (int hb = 0; hb < 2; ++hb) {  // value columns 64 hb .. 64 hb + 63: stage block hb
              float d[64];
              tc::ld64(acc + 64 * hb, d);
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const float2 y = mul2(P2, make_float2(d[2 * e], d[2 * e + 1]));
                d[2 * e] = y.x;
                d[2 * e + 1] = y.y;
              }
              const uint32_t row = hb * 16384 + r * 128;
#pragma unroll
              for (int q8 = 0; q8 < 8; ++q8) {
                const uint32_t off = row + ((q8 ^ (r & 7)) << 4);
                if (last) {  // the state is rounded once, here
                  *reinterpret_cast<uint4*>(st + off) =
                      make_uint4(pack_bf2(d[8 * q8], d[8 * q8 + 1]), pack_bf2(d[8 * q8 + 2], d[8 * q8 + 3]),
                                 pack_bf2(d[8 * q8 + 4], d[8 * q8 + 5]), pack_bf2(d[8 * q8 + 6], d[8 * q8 + 7]));
                } else {  // GEMM 1 operand of the next chunk: bf16 high and low parts
                  float y[8];
#pragma unroll
                  for (int e = 0; e < 8; ++e) y[e] = d[8 * q8 + e];
                  uint4 yh, yl;
                  split8(y, yh, yl);
                  *reinterpret_cast<uint4*>(st + off) = yh;
                  *reinterpret_cast<uint4*>(lo + off) = yl;
                }
              }
              if (!last) {  // S' (float32) stays in the accumulator for the next chunk
                tc::st32(acc + 64 * hb, *reinterpret_cast<const float(*)[32]>(d));
                tc::st32(acc + 64 * hb + 32, *reinterpret_cast<const float(*)[32]>(d + 32));
              }
            }
            tc::fence_before_sync();
            fence_proxy_async_smem();
            if (!last) {
              mbar_arrive(sready);
            } else if (!VERIFY) {
              if (!group_sync(ebar, (nstore++) & 1)) { run = false; break; }  // every row of S' is in the stage
              if (elected) {
                tma_store_3d(&map, st, 0, h * kD, slot);
                tma_store_3d(&map, st + 16384, 64, h * kD, slot);
                bulk_commit();
                pend = s;
              }
            }
          }
          mbar_arrive(&efree[b]);
          ++it;
          tok0 += nt;
          if (last) break;
        }
        ++L;
      }
    }
    if (elected) bulk_wait_all();  // the last stores are complete before the CTA exits
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::dealloc(taddr, TMEM_COLS);
  }
}

namespace {

template <bool VERIFY>
cudaError_t launch_spec_mma_variant(const SpecArgs& a, int sm_count, cudaStream_t s) {
  CUtensorMap map;
  if (!encode_state_map<__nv_bfloat16>(&map, a.state, a.H, a.num_slots, a.slot_stride)) return cudaErrorNotSupported;
  static std::atomic<bool> set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kda_spec_mma_kernel<VERIFY>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)MMA_SMEM);
    if (e != cudaSuccess) return e;
    set[dev].store(true, std::memory_order_release);
  }
  const int64_t units = (int64_t)a.N * a.H;
  const int grid = (int)(units < sm_count ? (units > 0 ? units : 1) : sm_count);
  return launch_pdl(kda_spec_mma_kernel<VERIFY>, dim3(grid), dim3(MMA_THREADS), MMA_SMEM, s, 1, a, map);
}

}  // namespace

cudaError_t launch_spec_mma(const SpecArgs& a, bool verify, int sm_count, cudaStream_t s) {
  return verify ? launch_spec_mma_variant<true>(a, sm_count, s) : launch_spec_mma_variant<false>(a, sm_count, s);
}

cudaError_t read_mma_error(unsigned int* flags, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(flags, g_kda_mma_error, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_kda_mma_error, &zero, sizeof(unsigned int));
}

}  // namespace kda

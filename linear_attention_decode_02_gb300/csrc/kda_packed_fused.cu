// Packed fused speculative decode (conv + SiLU + KDA + gated RMSNorm over
// T >= 1 token rows per sequence) with per-token checkpoints of both caches.
#include <cooperative_groups.h>

#include <algorithm>
#include <atomic>

#include "kda_launch.h"
#include "kda_packed_fused.h"
#include "kda_stream_common.cuh"

namespace cg = cooperative_groups;

namespace kda {

namespace {

// 16-byte global -> shared copy through L2 (cp.async.cg); completes at the
// next cp_async_wait_all of the issuing thread.
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst_smem))),
               "l"(src)
               : "memory");
}
// 4-byte global -> shared copy (cp.async.ca), same completion rule.
__device__ __forceinline__ void cp_async4(void* dst_smem, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst_smem))),
               "l"(src)
               : "memory");
}
// Shared -> global TMA tensor store of one box at coordinates (x, y, z),
// completing in the issuing thread's bulk group.  The lines are marked
// evict-first in L2 (nothing in the call reads a checkpoint back), as the
// streaming stores of the plain path are: H=12 N=128 76.9 -> 75.3 us.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], [%1], %5;" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(static_cast<uint32_t>(__cvta_generic_to_shared(src))), "r"(x), "r"(y), "r"(z), "l"(policy)
               : "memory");
}
// Hint: bring the 128-byte line holding `p` (a global address) into L2.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// Split cluster barrier: arrive (release: this thread's earlier memory
// accesses are ordered before the peers' accesses after their wait), then
// wait (acquire).  Every thread of every CTA of the cluster must arrive once
// before any of them can pass its wait.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait;" ::: "memory"); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Normalises one token's q and k (lane holds key rows 4*lane .. 4*lane+3),
// writes the per-row coefficient pairs (d k_hat, d q_hat) to cab and
// (d, k_hat) to cdk, and returns q_hat . k_hat.
__device__ __forceinline__ float token_coefficient_pairs(float4 q, float4 k, float4 d, int lane, float2* cab,
                                                         float2* cdk) {
  float qq = q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w;
  float kk = k.x * k.x + k.y * k.y + k.z * k.z + k.w * k.w;
  float qk = q.x * k.x + q.y * k.y + q.z * k.z + q.w * k.w;
  qq = warp_sum(qq);
  kk = warp_sum(kk);
  qk = warp_sum(qk);
  const float rq = rsqrtf(qq + kL2Eps);
  const float rk = rsqrtf(kk + kL2Eps);
  const float4 kh = make_float4(k.x * rk, k.y * rk, k.z * rk, k.w * rk);
  const float4 qh = make_float4(q.x * rq, q.y * rq, q.z * rq, q.w * rq);
  float4* ab = reinterpret_cast<float4*>(cab + 4 * lane);
  float4* dk = reinterpret_cast<float4*>(cdk + 4 * lane);
  ab[0] = make_float4(d.x * kh.x, d.x * qh.x, d.y * kh.y, d.y * qh.y);
  ab[1] = make_float4(d.z * kh.z, d.z * qh.z, d.w * kh.w, d.w * qh.w);
  dk[0] = make_float4(d.x, kh.x, d.y, kh.y);
  dk[1] = make_float4(d.z, kh.z, d.w, kh.w);
  return qk * rq * rk;
}

// Logistic function from the hardware exponential and an approximate
// reciprocal: 1 / (1 + e^-x), within a few float32 ulps of the rounded
// value; gives 0 where e^-x overflows.
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }

}  // namespace

// =====================================================================================
// One cluster of CL CTAs per (sequence, head); CTA `rank` owns the value
// columns [rank*W, rank*W + W).  Column form (ROWSPLIT false): warp w owns a
// strip of W/NW of them over all 128 key rows, so a token's reductions need
// no CTA barrier.  Row form (ROWSPLIT true, for the narrow slabs of large
// clusters): warp w owns key rows [16w, 16w+16) of all W columns and the
// warps' partial reductions meet in shared memory, one CTA barrier per
// token; every CTA keeps 8 warps for the conv and coefficient phases while
// each SM stores only W/128 of the state.  The per-row coefficients a
// token's reduction reads, (d k_hat, d q_hat), and those its update reads,
// (d, k_hat), sit in two arrays of pairs: one 8-byte shared load each.
// The state slab is loaded once from the start slot (the
// checkpoint of the last accepted token) and carried in float32 registers
// across the sequence's tokens; after each token it is stored to that
// token's checkpoint slot (rounded once if bf16), so a call moves one state
// read plus one state write per token.
//
// The prologue keeps dependent memory round trips to three: the parameters
// (conv taps, dt_bias, norm weight) are copied to shared memory
// asynchronously at entry, alongside the metadata loads (token range,
// accepted count, the first chunk's checkpoint slots); the chunk's
// activation rows (this CTA's slab of each of x's q, k and v sections, the
// raw gate, this slab of the output gate: 16-byte pieces) are staged as
// soon as the token range is known, alongside the start-slot lookup; then
// the state slab and the conv history of the CTA's channels are loaded.
//
// Tokens go in chunks of up to TC:
//  A. conv + SiLU of the chunk's tokens for the CTA's 3 W channels (its slab
//     of q, of k and of v; the tokens of a channel are independent given its
//     raw inputs) and their conv checkpoints, so every channel is computed
//     and written once per cluster; in a cluster the q and k activations go
//     to every CTA through distributed shared memory, and a cluster barrier
//     ends the phase;
//  B. the warps normalise q, k of the chunk's tokens, form the decays and
//     write the per-row coefficients (all 128 key rows, in every CTA);
//  C. every warp runs the chunk's tokens on its strip (column form: no CTA
//     barrier; with a bf16 state the column sums by reduce-scatter over the
//     row groups, then a gather of u): reduction, update, checkpoint store,
//     raw output.  Nothing else rides on this sequential chain;
//  D. one warp per token sums the squares of the slab's raw outputs.  With
//     one CTA per unit and a float32 state the same warp then writes the
//     token's gated output row.  Otherwise the sum goes to shared memory (in
//     a cluster: into every CTA, through distributed shared memory), and
//     after one barrier each CTA adds the CL sums locally and writes its
//     slab of the gated outputs.
// Grid slice n == N zeroes the padding token rows outside [qsl[0], qsl[N]).
//
// TMA (bf16 state, one CTA per unit, column form): a token's checkpoint goes
// from the warp's registers into its strip of shared memory (128 rows x CW
// columns, row-major: each store instruction fills 512 contiguous bytes) and
// leaves by a TMA tensor store of that strip, so the warp goes on to the next
// token while the store drains; before overwriting the strip the warp waits
// until the previous store has read it, and before exiting until its stores
// are complete.  Measured at H=12 T=5: N=128 80.4 -> 76.9 us, N=32 31.0 ->
// 28.0 us.  With a float32 state (8 KB strips) the same form is slower, 131
// vs 107 us at N=128, and two strips a warp (bf16) 83.8 us: both keep plain
// stores / one strip.
// =====================================================================================
template <typename StateT, int W, int NW, bool ROWSPLIT, bool TMA>
__global__ void __launch_bounds__(NW * 32, MinBlocks<NW>::value)
    kda_packed_fused_kernel(const PackedFusedArgs a, const __grid_constant__ CUtensorMap ckpt_map) {
  constexpr int NT = NW * 32, TC = 8;
  constexpr int CL = kD / W;                 // CTAs per (sequence, head)
  constexpr int CW = ROWSPLIT ? W : W / NW;  // columns of one warp's strip
  constexpr int NCH = 2 * kD + W;  // activations a CTA needs: all of q and k, this slab of v
  constexpr int NCV = 3 * W;       // conv channels a CTA computes: this slab of q, of k and of v
  constexpr int PT = W / 2 + 16;   // 16-byte staging pieces per token: the three slabs, the gate
  using G = Strip<StateT, CW>;
  // fragments per lane: all 128 rows (column form) or the warp's 16 (row form)
  constexpr int P = ROWSPLIT ? (kD / NW) / G::RPI : G::PASSES;
  static_assert(!ROWSPLIT || (kD / NW) % G::RPI == 0, "row form: a warp's rows must tile its passes");
  static_assert(CL * W == kD && (CL == 1 || CL == 2 || CL == 4 || CL == 8), "slabs must tile the 128 columns");
  static_assert(TC == 8, "the conv phase reads the chunk's checkpoint slots as two int4");
  static_assert(W % 8 == 0, "slabs are staged in 16-byte pieces");
  static_assert(!TMA || (CL == 1 && !ROWSPLIT), "TMA checkpoints: one CTA per unit, column form");
  constexpr uint32_t CKB = kD * CW * sizeof(StateT);  // one warp's checkpoint strip
  // The staged conv input (read in phase A) and the raw outputs (written in
  // phase C) share one buffer.
  // The conv's raw inputs of a channel in one column, oldest first: rows 0-2
  // the history, rows 3 .. 3 + nt - 1 the staged chunk rows (q | k | v slab).
  // The raw outputs (phase C) reuse the staged rows, never the history.
  constexpr int XO_BYTES = TC * NCV * 2 > TC * W * 4 ? TC * NCV * 2 : TC * W * 4;
  constexpr int HIST_BYTES = 3 * NCV * 2;
  static_assert(HIST_BYTES % 16 == 0, "staged rows must stay 16-byte aligned");
  __shared__ __align__(16) unsigned char s_hxo[HIST_BYTES + XO_BYTES];
  auto s_xh = reinterpret_cast<__nv_bfloat16 (*)[NCV]>(s_hxo);
  auto s_o = reinterpret_cast<float (*)[W]>(s_hxo + HIST_BYTES);  // raw outputs (slab)
  __shared__ float s_w[4][NCV];                         // conv taps of the CTA's channels
  __shared__ __align__(16) float s_dt[kD];              // dt_bias of this head
  __shared__ __align__(16) float s_nw[W];               // norm weight (slab)
  __shared__ __align__(16) __nv_bfloat16 s_gr[TC][kD];  // staged raw gates
  __shared__ __align__(16) __nv_bfloat16 s_og[TC][W];   // staged output-gate logits (slab)
  __shared__ __align__(16) float s_act[TC][NCH];        // SiLU(conv)
  __shared__ __align__(16) float2 s_cab[TC][kD];        // (d k_hat, d q_hat) per key row
  __shared__ __align__(16) float2 s_cdk[TC][kD];        // (d, k_hat) per key row
  __shared__ float2 s_tok[TC];                          // (beta, q_hat . k_hat)
  __shared__ __align__(16) int s_slot[TC];              // checkpoint slot, 0 = none
  __shared__ float s_part[2][CL][TC];                   // CTA r's sum of squares per token (2 chunk buffers)
  __shared__ float2 s_red[ROWSPLIT ? 2 : 1][ROWSPLIT ? NW : 1][ROWSPLIT ? W : 1];  // row form: (a, b) partials

  const int rank = CL == 1 ? 0 : (int)(blockIdx.x % CL);
  const int slab0 = rank * W;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int lcol = (ROWSPLIT ? 0 : warp * CW) + (lane % G::LPR) * G::VEC;  // column within the slab
  const int col0 = slab0 + lcol;
  const int row0 = (ROWSPLIT ? warp * (kD / NW) : 0) + lane / G::LPR;   // rows row0 + i*RPI, i < P
  extern __shared__ unsigned char s_dyn[];  // TMA: the warps' checkpoint strips, 128-byte aligned
  unsigned char* ck = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(s_dyn) + 127) & ~uintptr_t(127)) +
                      warp * CKB;
  const int HD = a.H * kD;
  // Local conv channel lc (this CTA's slab of q, then of k, then of v): its
  // section, its channel within the section and its column of s_act.
  auto sec_of = [](int lc) { return lc / W; };
  auto cis_of = [slab0](int lc) { return slab0 + lc % W; };
  auto act_of = [slab0](int lc) { return lc < 2 * W ? (lc / W) * kD + slab0 + lc % W : 2 * kD + lc - 2 * W; };
  __shared__ int4 s_pf;  // next unit: (start slot or 0, first token, end token, head)
  pdl_wait();
  pdl_launch_dependents();

  // Persistent: each cluster walks the units (sequence, head) with a stride
  // of the grid's cluster count; the padding slice is unit N*H .. (N+1)*H-1.
  const int num_units = (a.N + 1) * a.H;
  int chunk = 0;  // chunks this CTA has run, across its units: selects the sum-of-squares buffer
  const int unit_stride = gridDim.x / CL;
  for (int unit = blockIdx.x / CL; unit < num_units; unit += unit_stride) {
  const int h = unit % a.H;
  const int n = unit / a.H;
  __syncthreads();  // the previous unit is done with the shared arrays
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (int64_t)h * kD + slab0;
  auto zero_rows = [&](int lo, int hi) {  // this slab of output rows [lo, hi)
    for (int i = tid; i < (hi - lo) * (W / 4); i += NT) {
      const float z[4] = {0.f, 0.f, 0.f, 0.f};
      store_out<4>(out + (int64_t)(lo + i / (W / 4)) * a.o_rs + 4 * (i % (W / 4)), z);
    }
  };

  if (n == a.N) {  // padding token rows
    const int lo = min(max(__ldg(a.qsl), 0), a.R);
    const int hi = max(min(__ldg(a.qsl + a.N), a.R), lo);
    zero_rows(0, lo);
    zero_rows(hi, a.R);
    continue;
  }

  // Parameters first: they depend on nothing, so their copies overlap the
  // metadata loads below.
  for (int lc = tid; lc < NCV; lc += NT) {
    const float* w = a.conv_w + (int64_t)sec_of(lc) * 4 * HD + h * kD + cis_of(lc);
#pragma unroll
    for (int p = 0; p < 4; ++p) cp_async4(&s_w[p][lc], w + (int64_t)p * HD);
  }
  for (int i = tid; i < 32 + W / 4; i += NT) {
    if (i < 32) cp_async16(&s_dt[4 * i], a.dt_bias + h * kD + 4 * i);
    else cp_async16(&s_nw[4 * (i - 32)], a.norm_w + slab0 + 4 * (i - 32));
  }
  cp_async_commit();
  const float A = expf(__ldg(a.A_log + h));

  const int32_t* row_slots = a.idx + (int64_t)n * a.idx_rs;
  const int t0 = max(__ldg(a.qsl + n), 0);
  const int t1 = min(__ldg(a.qsl + n + 1), a.R);
  const int acc = __ldg(a.accepted + n);
  int slot = (tid < TC && tid < a.cols) ? __ldg(row_slots + tid) : 0;  // first chunk's checkpoints
  // The next unit this CTA runs: its metadata now, its slot during phase A.
  const int next = unit + unit_stride;
  const int next_n = next / a.H;
  int pf_t0 = 0, pf_t1 = 0, pf_acc = 0, pf_slot = 0;
  if (tid == 0 && next_n < a.N) {
    pf_t0 = max(__ldg(a.qsl + next_n), 0);
    pf_t1 = min(__ldg(a.qsl + next_n + 1), a.R);
    pf_acc = __ldg(a.accepted + next_n);
  }
  if (t1 <= t0) {  // empty sequence: nothing written
    cp_async_wait_all();
    continue;
  }
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(a.x);
  const __nv_bfloat16* gb = static_cast<const __nv_bfloat16*>(a.gate);
  const __nv_bfloat16* ogb = static_cast<const __nv_bfloat16*>(a.out_gate);

  auto stage = [&](int tc0, int nt) {
    for (int i = tid; i < nt * PT; i += NT) {
      const int j = i / PT, c = i % PT;
      const int64_t t = tc0 + j;
      const __nv_bfloat16* xr = xb + t * a.x_rs + h * kD;
      if (c < 3 * W / 8) {  // the q, k and v sections: this slab of each
        const int sec = c / (W / 8), part = c % (W / 8);
        cp_async16(&s_xh[3 + j][sec * W + part * 8], xr + (int64_t)sec * HD + slab0 + part * 8);
      } else if (c < 3 * W / 8 + 16) {
        const int part = c - 3 * W / 8;
        cp_async16(&s_gr[j][part * 8], gb + t * a.g_rs + (int64_t)h * a.g_hs + part * 8);
      } else {
        const int part = c - 3 * W / 8 - 16;
        cp_async16(&s_og[j][part * 8], ogb + t * a.og_rs + (int64_t)h * a.og_hs + slab0 + part * 8);
      }
    }
    cp_async_commit();
  };

  stage(t0, min(TC, t1 - t0));
  float braw = tid < min(TC, t1 - t0) ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.beta)[
                                            (int64_t)(t0 + tid) * a.b_rs + (int64_t)h * a.b_hs])
                                      : 0.f;
  const bool live_acc = acc >= 1 && acc <= a.cols;
  const int s0 = live_acc ? __ldg(row_slots + acc - 1) : 0;
  if (s0 <= 0 || s0 >= a.num_slots) {  // null sequence: zero its rows, touch no cache
    zero_rows(t0, t1);
    cp_async_wait_all();
    continue;
  }

  const int64_t head_off = (int64_t)h * kD * kD;
  float2 S[P][G::VEC / 2];  // float32 state fragments: rows row0 + i*RPI, columns col0..col0+VEC
  {
    const StateT* sp = static_cast<const StateT*>(a.state) + (int64_t)s0 * a.slot_stride + head_off;
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const typename Frag<StateT>::Raw r = Frag<StateT>::load(sp + (row0 + i * G::RPI) * kD + col0);
#pragma unroll
      for (int q = 0; q < G::VEC / 2; ++q) S[i][q] = Frag<StateT>::get2(r, q);
    }
  }

  __nv_bfloat16* cs = static_cast<__nv_bfloat16*>(a.conv_state);
  for (int lc = tid; lc < NCV; lc += NT) {
    const __nv_bfloat16* cp = cs + (int64_t)s0 * a.cs_slot_stride + sec_of(lc) * HD + h * kD + cis_of(lc);
#pragma unroll
    for (int p = 0; p < 3; ++p) s_xh[p][lc] = cp[p * a.cs_tap_stride];
  }
  // Cluster: a CTA reads and writes the conv cache of its own slab of each
  // section only; its q and k activations go to every peer's shared memory.
  // This arrive, with the wait before phase A, has every CTA of the cluster
  // running before the first distributed-shared-memory store.
  if constexpr (CL > 1) cluster_arrive();

  // The next unit this CTA runs, for its L2 prefetch: its start slot (loaded
  // before phase A) goes to shared memory, then every thread prefetches a
  // share of its lines.  With a bf16 state thread 0 publishes after phase B,
  // two phases after the slot load was issued, so no warp waits for that
  // load at a barrier (H=12 N=128 85.1 -> 82.3 us); with a float32 state
  // the earlier prefetch of the twice larger block wins (108 vs 110 us), and
  // it publishes after phase A.
  constexpr bool kLatePrefetch = sizeof(StateT) == 2;
  auto publish_next = [&] {
    s_pf = make_int4(pf_slot > 0 && pf_slot < a.num_slots ? pf_slot : 0, pf_t0, min(pf_t1, pf_t0 + TC), next % a.H);
  };
  auto prefetch_next = [&](int tc0) {
    if (tc0 == t0 && s_pf.x != 0) {
      const int4 pf = s_pf;
      const char* sb = reinterpret_cast<const char*>(static_cast<const StateT*>(a.state) +
                                                     (int64_t)pf.x * a.slot_stride + (int64_t)pf.w * kD * kD);
      constexpr int NL = kD * kD * (int)sizeof(StateT) / 128;  // 128-byte lines of a state block
      for (int i = rank * (NL / CL) + tid; i < (rank + 1) * (NL / CL); i += NT) prefetch_l2(sb + (int64_t)i * 128);
      if (rank == 0) {
        const int ntok = pf.z - pf.y;
        for (int i = tid; i < ntok * 10 + 18; i += NT) {
          const __nv_bfloat16* line;
          if (i < ntok * 10) {
            const int64_t t = pf.y + i / 10;
            const int c = i % 10;
            if (c < 6) line = xb + t * a.x_rs + (int64_t)(c >> 1) * HD + pf.w * kD + (c & 1) * 64;
            else if (c < 8) line = gb + t * a.g_rs + (int64_t)pf.w * a.g_hs + (c - 6) * 64;
            else line = ogb + t * a.og_rs + (int64_t)pf.w * a.og_hs + (c - 8) * 64;
          } else {
            const int c = i - ntok * 10;  // tap c / 6, section (c % 6) / 2, half c % 2
            line = cs + (int64_t)pf.x * a.cs_slot_stride + (int64_t)(c / 6) * a.cs_tap_stride +
                   (int64_t)((c % 6) >> 1) * HD + pf.w * kD + (c & 1) * 64;
          }
          prefetch_l2(line);
        }
      }
    }
  };

  for (int tc0 = t0; tc0 < t1; tc0 += TC) {
    const int nt = min(TC, t1 - tc0);
    const int p0 = tc0 - t0;  // position of the chunk's first token in its sequence
    if (tc0 != t0) {
      __syncthreads();  // previous chunk's epilogue done with the shared arrays
      stage(tc0, nt);
      if (tid < nt) {
        braw = __bfloat162float(
            static_cast<const __nv_bfloat16*>(a.beta)[(int64_t)(tc0 + tid) * a.b_rs + (int64_t)h * a.b_hs]);
        slot = p0 + tid < a.cols ? __ldg(row_slots + p0 + tid) : 0;
      }
    }
    cp_async_wait_all();
    if (tid < nt) {
      s_tok[tid].x = sigmoidf_(braw);
      s_slot[tid] = (slot > 0 && slot < a.num_slots) ? slot : 0;
    }
    __syncthreads();

    if (tid == 0 && tc0 == t0 && next_n < a.N && pf_t1 > pf_t0 && pf_acc >= 1 && pf_acc <= a.cols)
      pf_slot = __ldg(a.idx + (int64_t)next_n * a.idx_rs + pf_acc - 1);
    if constexpr (CL > 1) {
      if (tc0 == t0) cluster_wait();  // every peer is running
    }
    // ---- A: conv + SiLU and the conv checkpoints of this CTA's channels
    // Token j's conv reads raw rows j .. j+3 and leaves the history j+1 ..
    // j+3, so the chunk's (token, channel) items are independent: they are
    // spread evenly over the threads, tokens outer, the chunk's nt tokens
    // only.  In a cluster each q and k activation is written into every
    // CTA's s_act (its own included); the cluster barrier ending the phase
    // makes them visible.  A peer's reads of the previous chunk's
    // activations all precede the previous chunk's RMSNorm cluster barrier.
    for (int i = tid; i < nt * NCV; i += NT) {
      const int j = i / NCV, lc = i - j * NCV;
      float y = s_w[0][lc] * __bfloat162float(s_xh[j][lc]);
      y = fmaf(s_w[1][lc], __bfloat162float(s_xh[j + 1][lc]), y);
      y = fmaf(s_w[2][lc], __bfloat162float(s_xh[j + 2][lc]), y);
      y = fmaf(s_w[3][lc], __bfloat162float(s_xh[j + 3][lc]), y);
      const float act = y * sigmoid_fast(y);
      const int ac = act_of(lc);
      if constexpr (CL > 1) {
        if (lc < 2 * W) {
#pragma unroll
          for (int r = 0; r < CL; ++r) *cg::this_cluster().map_shared_rank(&s_act[j][ac], r) = act;
        } else {
          s_act[j][ac] = act;
        }
      } else {
        s_act[j][ac] = act;
      }
      const int sl = s_slot[j];
      if (sl != 0) {  // token j's conv checkpoint of this channel
        __nv_bfloat16* cp = cs + (int64_t)sl * a.cs_slot_stride + (int64_t)sec_of(lc) * HD + h * kD + cis_of(lc);
        cp[0] = s_xh[j + 1][lc];
        cp[a.cs_tap_stride] = s_xh[j + 2][lc];
        cp[2 * a.cs_tap_stride] = s_xh[j + 3][lc];
      }
    }
    // The next chunk's history, rows nt .. nt+2, held in registers until
    // every thread has read this chunk's rows (the barrier below).
    constexpr int HPT = (NCV + NT - 1) / NT;  // history channels per thread
    __nv_bfloat16 nh[HPT][3];
#pragma unroll
    for (int c = 0; c < HPT; ++c) {
      const int lc = tid + c * NT;
#pragma unroll
      for (int p = 0; p < 3; ++p) nh[c][p] = lc < NCV ? s_xh[nt + p][lc] : __float2bfloat16(0.f);
    }
    if constexpr (!kLatePrefetch) {
      if (tid == 0 && tc0 == t0) publish_next();
    }
    if constexpr (CL > 1) {
      cluster_arrive();  // this CTA's activations are written (release) ...
      cluster_wait();    // ... and every peer's (acquire)
    } else {
      __syncthreads();
    }
#pragma unroll
    for (int c = 0; c < HPT; ++c) {
      const int lc = tid + c * NT;
      if (lc < NCV) {
#pragma unroll
        for (int p = 0; p < 3; ++p) s_xh[p][lc] = nh[c][p];
      }
    }
    if constexpr (!kLatePrefetch) prefetch_next(tc0);

    // ---- B: per-token decays and coefficients
    for (int j = warp; j < nt; j += NW) {
      const float4 dtb = *reinterpret_cast<const float4*>(&s_dt[4 * lane]);
      const float4 q = *reinterpret_cast<const float4*>(&s_act[j][4 * lane]);
      const float4 k = *reinterpret_cast<const float4*>(&s_act[j][kD + 4 * lane]);
      const uint2 gr = *reinterpret_cast<const uint2*>(&s_gr[j][4 * lane]);
      const float4 d = make_float4(expf(log_decay(bf_lo(gr.x) + dtb.x, A, a.gate_mode, a.lower_bound)),
                                   expf(log_decay(bf_hi(gr.x) + dtb.y, A, a.gate_mode, a.lower_bound)),
                                   expf(log_decay(bf_lo(gr.y) + dtb.z, A, a.gate_mode, a.lower_bound)),
                                   expf(log_decay(bf_hi(gr.y) + dtb.w, A, a.gate_mode, a.lower_bound)));
      const float qk = token_coefficient_pairs(q, k, d, lane, s_cab[j], s_cdk[j]);
      if (lane == 0) s_tok[j].y = qk;
    }
    if constexpr (kLatePrefetch) {
      if (tid == 0 && tc0 == t0) publish_next();
    }
    __syncthreads();
    if constexpr (kLatePrefetch) prefetch_next(tc0);

    // ---- C: the chunk's tokens on this warp's fragments
    for (int j = 0; j < nt; ++j) {
      const float2 tk = s_tok[j];
      float2 a2[G::VEC / 2], b2[G::VEC / 2];
#pragma unroll
      for (int q = 0; q < G::VEC / 2; ++q) { a2[q] = make_float2(0.f, 0.f); b2[q] = make_float2(0.f, 0.f); }
#pragma unroll
      for (int i = 0; i < P; ++i) {
        const float2 c = s_cab[j][row0 + i * G::RPI];
        accumulate_row<G::VEC / 2>(make_float4(c.x, c.y, 0.f, 0.f), S[i], a2, b2);
      }
      float u[G::VEC], o[G::VEC];
      // Column form, bf16 state (16 row groups: 24 shuffles instead of 64;
      // measured 4 % faster at N=128, while fp32's 8 row groups gain nothing):
      // the lane of row group rg holds the total a_rg (rg < VEC: it forms u
      // for column rg) or b_{rg-VEC} (it forms o for that column with the u of
      // the lane VEC row groups below).  Then every lane gathers the VEC u.
      constexpr bool kScatter = !ROWSPLIT && sizeof(StateT) == 2;
      if constexpr (kScatter) {
        const int rg = lane / G::LPR;
        const float tot = strip_reduce_scatter<G>(a2, b2, rg);
        const float uc = rg < G::VEC ? tk.x * (s_act[j][2 * kD + lcol + rg] - tot) : 0.f;
        const float u_lo = __shfl_xor_sync(0xffffffffu, uc, G::LPR * G::VEC);
        if (rg >= G::VEC) s_o[j][lcol + rg - G::VEC] = a.scale * (tot + tk.y * u_lo);
#pragma unroll
        for (int c = 0; c < G::VEC; ++c) u[c] = __shfl_sync(0xffffffffu, uc, c * G::LPR + lane % G::LPR);
      } else {
        float acc_a[G::VEC], acc_b[G::VEC];
        strip_allreduce<G>(a2, b2, acc_a, acc_b);
        if constexpr (ROWSPLIT) {  // combine the warps' row partials
          if (lane < G::LPR) {
#pragma unroll
            for (int jj = 0; jj < G::VEC; ++jj) s_red[j & 1][warp][lcol + jj] = make_float2(acc_a[jj], acc_b[jj]);
          }
          __syncthreads();
#pragma unroll
          for (int jj = 0; jj < G::VEC; ++jj) {
            float ta = 0.f, tb = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
              const float2 r = s_red[j & 1][w][lcol + jj];
              ta += r.x;
              tb += r.y;
            }
            acc_a[jj] = ta;
            acc_b[jj] = tb;
          }
        }
#pragma unroll
        for (int jj = 0; jj < G::VEC; ++jj) {
          u[jj] = tk.x * (s_act[j][2 * kD + lcol + jj] - acc_a[jj]);
          o[jj] = a.scale * (acc_b[jj] + tk.y * u[jj]);
        }
      }
      float2 u2[G::VEC / 2];
      pairs_of<G::VEC>(u, u2);
#pragma unroll
      for (int i = 0; i < P; ++i) {
        const float2 c = s_cdk[j][row0 + i * G::RPI];
        update_row<G::VEC / 2>(c.x, c.y, S[i], u2, S[i]);
      }
      const int sl = s_slot[j];
      if (sl != 0) {
        if constexpr (TMA) {
          if (lane == 0) bulk_wait_read();  // the previous checkpoint has left the strip
          __syncwarp();
#pragma unroll
          for (int i = 0; i < P; ++i)
            *reinterpret_cast<typename Frag<StateT>::Raw*>(
                ck + ((row0 + i * G::RPI) * CW + (lane % G::LPR) * G::VEC) * sizeof(StateT)) = Frag<StateT>::pack2(S[i]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&ckpt_map, ck, warp * CW, h * kD, sl);
            bulk_commit();
          }
        } else {
          StateT* sp = static_cast<StateT*>(a.state) + (int64_t)sl * a.slot_stride + head_off;
#pragma unroll
          for (int i = 0; i < P; ++i)
            Frag<StateT>::store(sp + (row0 + i * G::RPI) * kD + col0, Frag<StateT>::pack2(S[i]));
        }
      }
      if constexpr (!kScatter) {
        // lanes of the first row of each strip hold distinct columns (row form: warp 0 only)
        if (lane < G::LPR && (!ROWSPLIT || warp == 0)) {
#pragma unroll
          for (int jj = 0; jj < G::VEC; ++jj) s_o[j][lcol + jj] = o[jj];
        }
      }
    }
    __syncthreads();
    // ---- D: gated RMSNorm, one warp per token: the sum of squares of the
    // slab's raw outputs.  With one CTA per unit and a float32 state the same
    // warp writes the token's output row (measured: fp32 N=128 1.7 % faster,
    // bf16 1.4 % slower than all threads writing after a barrier).
    constexpr bool kRowPerWarp = CL == 1 && sizeof(StateT) == 4;
    auto gated_row = [&](int j, int c4, float rinv) {
      const float4 o4 = *reinterpret_cast<const float4*>(&s_o[j][c4]);
      const uint2 g2 = *reinterpret_cast<const uint2*>(&s_og[j][c4]);
      const float4 nw = *reinterpret_cast<const float4*>(&s_nw[c4]);
      float y[4] = {o4.x * rinv * nw.x * sigmoid_fast(bf_lo(g2.x)), o4.y * rinv * nw.y * sigmoid_fast(bf_hi(g2.x)),
                    o4.z * rinv * nw.z * sigmoid_fast(bf_lo(g2.y)), o4.w * rinv * nw.w * sigmoid_fast(bf_hi(g2.y))};
      store_out<4>(out + (int64_t)(tc0 + j) * a.o_rs + c4, y);
    };
    const int pb = chunk & 1;
    ++chunk;
    for (int j = warp; j < nt; j += NW) {
      float ss = 0.f;
#pragma unroll
      for (int c = lane; c < W; c += 32) ss = fmaf(s_o[j][c], s_o[j][c], ss);
      ss = warp_sum(ss);
      if constexpr (CL > 1) {
        // sent to every CTA of the cluster; the chunk buffers alternate, so a
        // fast CTA's next chunk never overwrites sums a peer is still reading
        if (lane < CL) *cg::this_cluster().map_shared_rank(&s_part[pb][rank][j], lane) = ss;
      } else if constexpr (kRowPerWarp) {
        const float rinv = rsqrtf(ss * (1.f / kD) + a.norm_eps);
#pragma unroll
        for (int c4 = 4 * lane; c4 < W; c4 += 128) gated_row(j, c4, rinv);
      } else {
        if (lane == 0) s_part[pb][0][j] = ss;
      }
    }
    if constexpr (!kRowPerWarp) {
      if constexpr (CL > 1) {
        cg::this_cluster().sync();  // every CTA's sums have arrived in every CTA
      } else {
        __syncthreads();
      }
      for (int i = tid; i < nt * (W / 4); i += NT) {
        const int j = i / (W / 4), c4 = 4 * (i % (W / 4));
        float tot = 0.f;
#pragma unroll
        for (int r = 0; r < CL; ++r) tot += s_part[pb][r][j];
        gated_row(j, c4, rsqrtf(tot * (1.f / kD) + a.norm_eps));
      }
    }
  }
  }  // units
  if constexpr (TMA) {
    if (lane == 0) bulk_wait_all();  // the strips stay in use until the stores have read them
  }
}

// The pool [num_slots][H*128 rows][128 columns] as a 3-d tensor map whose box
// is one warp's checkpoint strip: `cols` columns x 128 rows of one (slot,
// head) state, unswizzled.  The map of the last pool seen by this host
// thread is kept, so a serving loop encodes it once.
template <typename StateT>
bool ckpt_map_for(CUtensorMap* map, void* state, int H, int num_slots, int64_t slot_stride, int cols) {
  struct Key {
    void* state;
    int H, num_slots, cols, bytes;
    int64_t slot_stride;
  };
  thread_local Key last{nullptr, 0, 0, 0, 0, 0};
  thread_local CUtensorMap last_map;
  const Key k{state, H, num_slots, cols, (int)sizeof(StateT), slot_stride};
  if (last.state == k.state && last.H == k.H && last.num_slots == k.num_slots && last.cols == k.cols &&
      last.bytes == k.bytes && last.slot_stride == k.slot_stride) {
    *map = last_map;
    return true;
  }
  EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H * kD, (cuuint64_t)num_slots};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * sizeof(StateT), (cuuint64_t)slot_stride * sizeof(StateT)};
  const cuuint32_t box[3] = {(cuuint32_t)cols, (cuuint32_t)kD, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(map, sizeof(StateT) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, state, dims,
          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  last = k;
  last_map = *map;
  return true;
}

template <typename StateT, int W, int NW, bool ROWSPLIT, bool TMA>
cudaError_t launch_packed_fused_variant(const PackedFusedArgs& a, int sms, cudaStream_t s) {
  constexpr int CL = kD / W;
  constexpr int CW = ROWSPLIT ? W : W / NW;
  auto kernel = kda_packed_fused_kernel<StateT, W, NW, ROWSPLIT, TMA>;
  CUtensorMap map{};
  constexpr size_t smem = TMA ? (size_t)NW * kD * CW * sizeof(StateT) + 128 : 0;
  if constexpr (TMA) {
    // a pool the tensor map cannot describe takes the plain-store kernel
    if (!ckpt_map_for<StateT>(&map, a.state, a.H, a.num_slots, a.slot_stride, CW))
      return launch_packed_fused_variant<StateT, W, NW, ROWSPLIT, false>(a, sms, s);
    static std::atomic<bool> set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !set[dev].load(std::memory_order_acquire)) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      set[dev].store(true, std::memory_order_release);
    }
  }
  const int64_t units = (int64_t)(a.N + 1) * a.H;  // unit N*H.. is the padding slice
  int64_t clusters = units;
  if (CL == 1) {  // persistent: as many CTAs as fit on the device at once
    static const int per_sm = [&] {
      int b = 0;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, NW * 32, smem) == cudaSuccess && b > 0 ? b : 1;
    }();
    clusters = std::min<int64_t>(units, (int64_t)per_sm * sms);
  }
  return launch_pdl(kernel, dim3((unsigned)(clusters * CL)), dim3(NW * 32), smem, s, CL, a, map);
}

template <typename StateT>
cudaError_t launch_packed_fused_typed(const PackedFusedArgs& a, int cluster, int sms, cudaStream_t s) {
  switch (cluster) {
    case 1:  // TMA checkpoint stores with a bf16 state (see the kernel's comment)
      return launch_packed_fused_variant<StateT, 128, 8, false, sizeof(StateT) == 2>(a, sms, s);
    case 2: return launch_packed_fused_variant<StateT, 64, 4, false, false>(a, sms, s);
    case 4: return launch_packed_fused_variant<StateT, 32, 8, true, false>(a, sms, s);
    case 8: return launch_packed_fused_variant<StateT, 16, 8, true, false>(a, sms, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_packed_fused(const PackedFusedArgs& a, int state_dtype, int cluster, int sms, cudaStream_t s) {
  if (state_dtype == KDA_DT_F32) return launch_packed_fused_typed<float>(a, cluster, sms, s);
  return launch_packed_fused_typed<__nv_bfloat16>(a, cluster, sms, s);
}

}  // namespace kda

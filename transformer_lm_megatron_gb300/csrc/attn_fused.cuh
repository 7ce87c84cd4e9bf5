// Fused causal attention core of the self-attention block's forward, for one GB300
// (sm_103a): per (sequence, head) and tile of 128 queries,
//
//   S = Q K^T / sqrt(d)   (keys <= query),   P = softmax(S),   O_head = P V
//
// with S kept on chip.  The block's heads are the column split of the fused QKV
// projection (tensor slicing, "STRONGHOLD" slides items 7-8, read for attention
// as in the block's header); each head attends causally within its sequence (a
// left-to-right decoder with 128 heads: jiqizhixin article on MT-NLG).
//
// Two passes over the key tiles 0 .. i of query tile i:
//   pass 1  S_j = Q K_j^T into tensor memory; each query row keeps its running
//           maximum m and sum l = sum_k exp(s_k - m) (rescaled when m grows);
//   pass 2  S_j again; P_j = exp(S_j - m) / l, rounded to bf16, goes to shared
//           memory, where it is the A operand of O += P_j V_j, and to global memory
//           (the backward reads P); the O accumulator in tensor memory then holds
//           the final O, with no rescaling.
// P is written as exact zeros above the causal diagonal, as the unfused path does.
//
// Warp roles (320 threads, one CTA per SM, persistent over the work items, the
// items with the most key tiles first):
//   warp 0     TMA producer: Q (once per item), then K_0 .. K_i (pass 1), then
//              K_0, K_1, V_0, K_2, V_1, ... (pass 2) through a 2-slot ring.
//   warp 1     TMEM owner and MMA issuer (one thread): S into two 128-column
//              buffers; in pass 2 S_{j+1} is issued before O += P_j V_j so the
//              softmax of one tile overlaps the products of the next.
//   warps 2-9  one query row per thread (TMEM lane quarter warp % 4), two warps
//              per row, each on 64 of the 128 keys of every tile (their row
//              statistics merged once per item), then half of the zeros above the
//              diagonal and half of the bf16 O columns.
// Every wait is bounded; on timeout the kernel records kStatusTimeout in the
// status word and stops.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace gbmlp {

constexpr int kFaTile = 128;                         // queries per tile; keys per key tile
constexpr int kFaMaxAtoms = 3;                       // head size d <= 192 (64 columns per atom)
constexpr uint32_t kFaAtomBytes = 128 * 128;         // 128 rows x 64 bf16
constexpr uint32_t kFaTileBytes = kFaMaxAtoms * kFaAtomBytes;   // a Q, K or V tile: 48 KB
constexpr int kFaStages = 2;                         // K / V ring
constexpr uint32_t kFaPBytes = 2 * kFaAtomBytes;     // P tile, 128 x 128 bf16
constexpr uint32_t kFaOStageBytes = 32 * 32 * 2;     // one 32 x 32 bf16 output box
constexpr int kFaSoftmaxWarps = 8;                   // two per TMEM lane quarter
constexpr int kFaThreads = 64 + 32 * kFaSoftmaxWarps;
constexpr uint32_t kFaTmemCols = 512;                // S buffers at 0 and 128, O at 256
// Q, the K/V ring, two P buffers (which also stage the O stores at the end of an
// item), barriers, and the softmax halves' partial maxima and sums.
constexpr size_t kFaSmemBytes = (size_t)kFaTileBytes * (1 + kFaStages) + 2 * kFaPBytes + 1024 /*align*/ +
                                256 /*barriers*/ + 2 * 2 * 128 * 2 * sizeof(float);
static_assert(kFaSmemBytes <= 232448, "smem budget");
static_assert(2 * kFaOStageBytes <= 32 * 128, "O staging fits in a warp's rows of a P buffer");
constexpr float kLog2e = 1.4426950408889634f;      // log2(e): exp(x) = 2^(x log2 e)

// 2^x with the hardware approximation (ex2.approx, flush-to-zero); 2^-inf = 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct FaParams {
  int L;          // sequence length (keys and queries per sequence)
  int nh;         // heads
  int ns;         // sequences
  int d;          // head size
  int d_pad;      // d rounded up to 16 (the N of O += P V)
  int n_atoms;    // ceil(d_pad / 64)
  float alpha;    // 1 / sqrt(d)
  uint16_t* P;    // [ns, nh, L, L] bf16
};

// maps: mQ, mK (box 64 x 128), mV (box 64 x 64) over QKV viewed as
// (d, L, nh, ns); mP (box 64 x 32) over P as (L, L, nh, ns); mO (box 32 x 32,
// 64-byte swizzle) over O as (d, L, nh, ns).
__global__ void __launch_bounds__(kFaThreads, 1)
    k_attn_fwd_fused(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                     const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mP,
                     const __grid_constant__ CUtensorMap mO, FaParams fp, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = sQ + kFaTileBytes;
  uint8_t* sP = sRing + kFaStages * kFaTileBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sP + 2 * kFaPBytes);
  uint64_t* q_full = bar;
  uint64_t* q_empty = bar + 1;
  uint64_t* kv_full = bar + 2;                 // [kFaStages]
  uint64_t* kv_empty = kv_full + kFaStages;    // [kFaStages]
  uint64_t* s_full = kv_empty + kFaStages;     // [2]
  uint64_t* s_empty = s_full + 2;              // [2]
  uint64_t* p_full = s_empty + 2;              // [2]
  uint64_t* p_empty = p_full + 2;              // [2]
  uint64_t* o_full = p_empty + 2;
  uint64_t* o_empty = o_full + 1;
  uint64_t* merged = o_empty + 1;              // the softmax warps' row statistics are in shared memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(merged + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_qt = (fp.L + kFaTile - 1) / kFaTile;
  const int heads = fp.nh * fp.ns;
  const int num_items = n_qt * heads;
  const uint32_t tile_tx = (uint32_t)fp.n_atoms * kFaAtomBytes;   // bytes of one Q, K or V tile

  __shared__ int s_skip;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kFaStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_empty[b], kFaSoftmaxWarps);   // every softmax warp reads its half of each S tile
      mbar_init(&p_full[b], kFaSoftmaxWarps);
      mbar_init(&p_empty[b], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(o_empty, kFaSoftmaxWarps);
    mbar_init(merged, kFaSoftmaxWarps);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mQ);
    tma_prefetch_desc(&mK);
    tma_prefetch_desc(&mV);
    tma_prefetch_desc(&mP);
    tma_prefetch_desc(&mO);
  }
  if (warp == 1) {
    tmem_alloc<false>(tmem_slot, kFaTmemCols);
    tmem_relinquish<false>();
  }
  grid_dependency_wait();
  grid_launch_dependents();
  if (threadIdx.x == 0) s_skip = (status != nullptr && *reinterpret_cast<volatile int*>(status) != 0) ? 1 : 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int item_end = s_skip ? 0 : num_items;

  // item -> (query tile, head, sequence): the tiles with the most key tiles first
  auto decode = [&](int item, int& qt, int& hb, int& sb) {
    qt = n_qt - 1 - item / heads;
    const int r = item % heads;
    hb = r % fp.nh;
    sb = r / fp.nh;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t kv = 0;  // ring uses so far
      bool ok = true;
      uint32_t n_item = 0;
      for (int item = blockIdx.x; item < item_end && ok; item += gridDim.x, ++n_item) {
        int qt, hb, sb;
        decode(item, qt, hb, sb);
        const int nkv = qt + 1;
        const int q0 = qt * kFaTile;
        if (!mbar_wait(q_empty, (n_item & 1) ^ 1)) {
          record_status(status, kStatusTimeout, 20);
          break;
        }
        mbar_arrive_expect_tx(q_full, tile_tx);
        for (int a = 0; a < fp.n_atoms; ++a) tma_load_4d(sQ + a * kFaAtomBytes, &mQ, q_full, 64 * a, q0, hb, sb);
        // pass 1: K_0 .. K_{nkv-1}; pass 2: K_0, then K_{j+1} (if any) and V_j for each j
        auto load_k = [&](int j) -> bool {
          const int s = (int)(kv % kFaStages);
          if (!mbar_wait(&kv_empty[s], ((kv / kFaStages) & 1) ^ 1)) return false;
          uint8_t* dst = sRing + s * kFaTileBytes;
          mbar_arrive_expect_tx(&kv_full[s], tile_tx);
          for (int a = 0; a < fp.n_atoms; ++a)
            tma_load_4d(dst + a * kFaAtomBytes, &mK, &kv_full[s], 64 * a, j * kFaTile, hb, sb);
          ++kv;
          return true;
        };
        auto load_v = [&](int j) -> bool {
          const int s = (int)(kv % kFaStages);
          if (!mbar_wait(&kv_empty[s], ((kv / kFaStages) & 1) ^ 1)) return false;
          uint8_t* dst = sRing + s * kFaTileBytes;
          mbar_arrive_expect_tx(&kv_full[s], tile_tx);
          // MN-major B operand of O += P V: two halves of 64 keys, each n_atoms chunks of 64 head columns
          for (int hk = 0; hk < 2; ++hk)
            for (int c = 0; c < fp.n_atoms; ++c)
              tma_load_4d(dst + (hk * fp.n_atoms + c) * 8192, &mV, &kv_full[s], 64 * c, j * kFaTile + 64 * hk, hb,
                          sb);
          ++kv;
          return true;
        };
        for (int j = 0; j < nkv && ok; ++j) ok = load_k(j);
        if (ok) ok = load_k(0);
        for (int j = 0; j < nkv && ok; ++j) {
          if (j + 1 < nkv) ok = load_k(j + 1);
          if (ok) ok = load_v(j);
        }
        if (!ok) record_status(status, kStatusTimeout, 21);
      }
      // Drain: every copy this CTA issued has landed before the CTA may exit (the
      // last use of each barrier completes the phase of parity (uses - 1) & 1).
      if (n_item > 0 && !mbar_wait(q_full, (n_item - 1) & 1)) record_status(status, kStatusTimeout, 24);
      for (uint32_t s = 0; s < (uint32_t)kFaStages; ++s) {
        const uint32_t uses = kv / kFaStages + (s < kv % kFaStages ? 1u : 0u);
        if (uses > 0 && !mbar_wait(&kv_full[s], (uses - 1) & 1)) record_status(status, kStatusTimeout, 25);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc_s = make_idesc_bf16(kFaTile, kFaTile, false, false);
      const uint32_t idesc_o = make_idesc_bf16(kFaTile, fp.d_pad, false, true);
      const int nk_s = fp.d_pad / 16;  // k-steps of S = Q K^T
      uint32_t kv = 0, sc = 0, pc = 0;
      bool ok = true;
      uint32_t n_item = 0;
      auto wait_kv = [&]() -> uint8_t* {
        const int s = (int)(kv % kFaStages);
        if (!mbar_wait(&kv_full[s], (kv / kFaStages) & 1)) return nullptr;
        tc_fence_after();
        return sRing + s * kFaTileBytes;
      };
      auto release_kv = [&]() {
        umma_commit(&kv_empty[kv % kFaStages]);
        ++kv;
      };
      // S_j = Q K_j^T into S buffer sc % 2
      auto issue_s = [&]() -> bool {
        uint8_t* kt = wait_kv();
        if (kt == nullptr) return false;
        const int b = (int)(sc & 1);
        if (!mbar_wait(&s_empty[b], ((sc >> 1) & 1) ^ 1)) return false;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(b * kFaTile);
        const uint32_t qb = smem_u32(sQ), kb = smem_u32(kt);
        for (int kk = 0; kk < nk_s; ++kk) {
          const uint32_t off = (uint32_t)(kk >> 2) * kFaAtomBytes + (uint32_t)(kk & 3) * 32;
          umma_bf16(d_tmem, make_sdesc_sw128(qb + off, 16, 1024), make_sdesc_sw128(kb + off, 16, 1024), idesc_s,
                    kk > 0 ? 1u : 0u);
        }
        release_kv();
        umma_commit(&s_full[b]);
        ++sc;
        return true;
      };
      // O (+)= P_j V_j
      auto issue_o = [&](bool first) -> bool {
        uint8_t* vt = wait_kv();
        if (vt == nullptr) return false;
        const int b = (int)(pc & 1);
        if (!mbar_wait(&p_full[b], (pc >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t o_tmem = tmem_base + 256u;
        const uint32_t pb = smem_u32(sP + b * kFaPBytes), vb = smem_u32(vt);
        for (int kk = 0; kk < kFaTile / 16; ++kk) {
          const uint32_t aoff = (uint32_t)(kk >> 2) * kFaAtomBytes + (uint32_t)(kk & 3) * 32;
          const uint32_t boff = (uint32_t)(kk >> 2) * (uint32_t)fp.n_atoms * 8192u + (uint32_t)(kk & 3) * 2048u;
          umma_bf16(o_tmem, make_sdesc_sw128(pb + aoff, 16, 1024), make_sdesc_sw128(vb + boff, 8192, 1024), idesc_o,
                    (first && kk == 0) ? 0u : 1u);
        }
        release_kv();
        umma_commit(&p_empty[b]);
        ++pc;
        return true;
      };
      for (int item = blockIdx.x; item < item_end && ok; item += gridDim.x, ++n_item) {
        int qt, hb, sb;
        decode(item, qt, hb, sb);
        const int nkv = qt + 1;
        if (!mbar_wait(q_full, n_item & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int j = 0; j < nkv && ok; ++j) ok = issue_s();          // pass 1
        if (ok) ok = issue_s();                                       // pass 2: S_0
        if (ok && nkv == 1) umma_commit(q_empty);
        if (ok && !mbar_wait(o_empty, (n_item & 1) ^ 1)) ok = false;  // the previous item's O has been read
        tc_fence_after();
        for (int j = 0; j < nkv && ok; ++j) {
          if (j + 1 < nkv) {
            ok = issue_s();                                           // S_{j+1} ahead of O += P_j V_j
            if (ok && j + 2 == nkv) umma_commit(q_empty);             // Q read for the last time
          }
          if (ok) ok = issue_o(j == 0);
        }
        if (ok) umma_commit(o_full);
      }
      if (!ok) record_status(status, kStatusTimeout, 22);
    }
  } else {
    // -------------------------------------------------------------- softmax / epilogue
    // Two warps per TMEM lane quarter: the warp of half h takes keys 64 h .. 64 h + 63
    // of every key tile.  Pass 1 gives each half a partial maximum and sum per row,
    // merged through shared memory; pass 2 writes its half of every P tile; the O
    // columns are shared out by 32-column block.
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r_in = quarter * 32 + lane;                  // query row within the tile
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    float* s_ml = reinterpret_cast<float*>(tmem_slot + 4);  // [2 items][2 halves][128 rows][m, l]
    const float al = fp.alpha * kLog2e;                     // scores in units of log2
    uint32_t sc = 0, pc = 0, n_out = 0;
    bool ok = true;
    uint32_t n_item = 0;
    for (int item = blockIdx.x; item < item_end && ok; item += gridDim.x, ++n_item) {
      int qt, hb, sb;
      decode(item, qt, hb, sb);
      const int nkv = qt + 1;
      // pass 1: the running maximum (log2 units) and sum of the row over this half's
      // 64 keys of every key tile
      float m = -INFINITY, l = 0.0f;
      for (int j = 0; j < nkv && ok; ++j, ++sc) {
        const int b = (int)(sc & 1);
        if (!(ok = mbar_wait(&s_full[b], (sc >> 1) & 1))) break;
        tc_fence_after();
        const uint32_t t_s = t_lane + (uint32_t)(b * kFaTile + 64 * half);
        const bool diag = j == qt;
        uint32_t r[2][32];
        tmem_ld_32x32b_x32(t_s, r[0]);
        tmem_ld_32x32b_x32(t_s + 32, r[1]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[b]);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int c0 = 64 * half + 32 * c;
          float mx = -INFINITY;
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float v = (diag && c0 + k > r_in) ? -INFINITY : al * __uint_as_float(r[c][k]);
            r[c][k] = __float_as_uint(v);
            mx = fmaxf(mx, v);
          }
          const float m_new = fmaxf(m, mx);
          const float m_ref = m_new == -INFINITY ? 0.0f : m_new;   // a block with every key masked adds 0
          float sum = 0.0f;
#pragma unroll
          for (int k = 0; k < 32; ++k) sum += ex2_approx(__uint_as_float(r[c][k]) - m_ref);
          l = (m == -INFINITY ? 0.0f : l * ex2_approx(m - m_new)) + sum;
          m = m_new;
        }
      }
      if (!ok) break;
      // merge the two halves (the same expression, in the same order, in both),
      // through one of two buffers by item parity
      float* ml = s_ml + (n_item & 1) * (2 * 128 * 2);
      ml[(half * 128 + r_in) * 2] = m;
      ml[(half * 128 + r_in) * 2 + 1] = l;
      // every softmax warp has written its statistics (a bounded wait, like every other:
      // a warp that gave up earlier never arrives, and the others give up in turn)
      __syncwarp();
      if (lane == 0) mbar_arrive(merged);
      if (!(ok = mbar_wait(merged, n_item & 1))) break;
      const float m0 = ml[r_in * 2], l0 = ml[r_in * 2 + 1];
      const float m1 = ml[(128 + r_in) * 2], l1 = ml[(128 + r_in) * 2 + 1];
      m = fmaxf(m0, m1);
      l = (m0 == -INFINITY ? 0.0f : l0 * ex2_approx(m0 - m)) + (m1 == -INFINITY ? 0.0f : l1 * ex2_approx(m1 - m));
      const float inv = 1.0f / l;
      // pass 2: this half's 64 columns of P_j = exp(S_j - max) / sum, to shared memory
      // (operand of O += P V) and to P
      for (int j = 0; j < nkv && ok; ++j, ++sc, ++pc) {
        const int b = (int)(sc & 1);
        const int pb = (int)(pc & 1);
        if (!(ok = mbar_wait(&s_full[b], (sc >> 1) & 1))) break;
        tc_fence_after();
        const uint32_t t_s = t_lane + (uint32_t)(b * kFaTile + 64 * half);
        uint32_t r[2][32];
        tmem_ld_32x32b_x32(t_s, r[0]);
        tmem_ld_32x32b_x32(t_s + 32, r[1]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[b]);
        // this warp's rows of the P buffer are free once the products that read it
        // are done and this warp's store of them (or of O) has read them
        if (!(ok = mbar_wait(&p_empty[pb], ((pc >> 1) & 1) ^ 1))) break;
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        uint8_t* atom = sP + pb * kFaPBytes + half * kFaAtomBytes;
        uint8_t* row = atom + r_in * 128;
        const bool diag = j == qt;
#pragma unroll
        for (int g = 0; g < 8; ++g) {         // keys 64 half + 8 g .. + 7: chunk g ^ (r_in % 8) of the atom
          uint32_t pk[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int k0 = 8 * g + 2 * k, k1 = k0 + 1;    // 0 .. 63 within the half
            const float s0 = __uint_as_float(r[k0 >> 5][k0 & 31]), s1 = __uint_as_float(r[k1 >> 5][k1 & 31]);
            const float p0 = (diag && 64 * half + k0 > r_in) ? 0.0f : ex2_approx(fmaf(s0, al, -m)) * inv;
            const float p1 = (diag && 64 * half + k1 > r_in) ? 0.0f : ex2_approx(fmaf(s1, al, -m)) * inv;
            pk[k] = pack_bf16x2(p0, p1);
          }
          *reinterpret_cast<uint4*>(row + ((g ^ (r_in & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_4d(&mP, atom + quarter * 32 * 128, j * kFaTile + 64 * half, qt * kFaTile + quarter * 32, hb, sb);
          bulk_commit();
          mbar_arrive(&p_full[pb]);
        }
      }
      if (!ok) break;
      // zeros above the diagonal: keys (qt + 1) * 128 .. L - 1 of this warp's rows
      // (while the last O += P V runs)
      {
        const int c_begin = nkv * kFaTile;
        const int z = fp.L - c_begin;
        if (z > 0) {
          for (int rr = half; rr < 32; rr += 2) {
            const int qq = qt * kFaTile + quarter * 32 + rr;
            if (qq >= fp.L) break;
            uint16_t* prow = fp.P + (((int64_t)sb * fp.nh + hb) * fp.L + qq) * (int64_t)fp.L + c_begin;
            for (int c = lane * 8; c < z; c += 256) *reinterpret_cast<uint4*>(prow + c) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      // this warp's P stores have read its rows of the first P buffer, which now stage O
      if (lane == 0) bulk_wait_read<0>();
      __syncwarp();
      if (!(ok = mbar_wait(o_full, n_item & 1))) break;
      tc_fence_after();
      // O: the accumulator is final; bf16 through 32 x 32 boxes, the column blocks
      // shared out between the halves, staged in this warp's rows of the first P buffer
      uint8_t* my_o = sP + half * kFaAtomBytes + quarter * 32 * 128;
      for (int c0 = 32 * half; c0 < fp.d_pad; c0 += 64) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_lane + 256u + (uint32_t)c0, r);
        tmem_ld_wait();
        if (c0 >= fp.d) continue;
        uint8_t* box = my_o + (n_out & 1) * kFaOStageBytes;
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint32_t off = lane * 64 + ((g ^ ((lane >> 1) & 3)) << 4);
          *reinterpret_cast<uint4*>(box + off) =
              make_uint4(pack_bf16x2(__uint_as_float(r[8 * g]), __uint_as_float(r[8 * g + 1])),
                         pack_bf16x2(__uint_as_float(r[8 * g + 2]), __uint_as_float(r[8 * g + 3])),
                         pack_bf16x2(__uint_as_float(r[8 * g + 4]), __uint_as_float(r[8 * g + 5])),
                         pack_bf16x2(__uint_as_float(r[8 * g + 6]), __uint_as_float(r[8 * g + 7])));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_4d(&mO, box, c0, qt * kFaTile + quarter * 32, hb, sb);
          bulk_commit();
        }
        ++n_out;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
    }
    if (!ok) record_status(status, kStatusTimeout, 23);
    if (lane == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<false>(tmem_base, kFaTmemCols);
  }
}

}  // namespace gbmlp

namespace gbmlp {

// ---------------------------------------------------------------------------
// Fused causal attention core of the backward, per (sequence, head) and tile j of
// 128 keys, over the query tiles i = j .. last (the keys of tile j see only those):
//
//   dP = dO_i V_j^T                        (tensor memory, a query row per lane)
//   dV_j += P_ij^T dO_i                    (tensor memory, fp32)
//   dS = P_ij (dP - delta_i) / sqrt(d), bf16, one query row per thread
//   dK_j += dS^T Q_i                       (tensor memory, fp32)
//
// with delta_i = rowsum(dO_i * O_i) given (k_attn_delta), the stored bf16 P of the
// forward, and dS written to global memory for dQ = dS K (a batched GEMM).  dK_j
// and dV_j go to dQKV in bf16.
// Every operand tile is loaded once, as 64-column swizzle atoms of 128 rows: such
// an atom is also two stacked MN-major chunks of 64 rows, so the same bytes serve
// as a K-major operand (dO and V for dP) and as an MN-major one (P and dO for dV,
// dS and Q for dK).
// Warps: 0 TMA producer, 1 TMEM owner and MMA issuer, 2-9 one query row per thread,
// two warps per row (TMEM lane quarter), each on half of the 128 keys of a tile.
// TMEM: dV at columns 0.., dK at 192.., dP at 384 .. 511.
// ---------------------------------------------------------------------------
constexpr int kFbRowWarps = 8;          // two per TMEM lane quarter, each on 64 of a tile's 128 keys
constexpr int kFbThreads = 64 + 32 * kFbRowWarps;
constexpr size_t kFbSmemBytes = (size_t)kFaTileBytes * 3 /* V, dO, Q */ + 2 * kFaPBytes /* P, dS^T */ +
                                kFaTile * sizeof(float) /* delta */ + 1024 /*align*/ + 256 /*barriers*/;
static_assert(kFbSmemBytes <= 232448, "smem budget");

struct FbParams {
  int L, nh, ns, d, d_pad, n_atoms;
  float alpha;     // 1 / sqrt(d)
  uint16_t* dS;    // [ns, nh, L queries, L keys] bf16
};

__global__ void __launch_bounds__(kFbThreads, 1)
    k_attn_bwd_fused(const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mQ,
                     const __grid_constant__ CUtensorMap mdO, const __grid_constant__ CUtensorMap mP,
                     const __grid_constant__ CUtensorMap mDelta, const __grid_constant__ CUtensorMap mDS,
                     const __grid_constant__ CUtensorMap mdK, const __grid_constant__ CUtensorMap mdV, FbParams fp,
                     int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sV = smem;
  uint8_t* sdO = sV + kFaTileBytes;
  uint8_t* sQ = sdO + kFaTileBytes;
  uint8_t* sP = sQ + kFaTileBytes;
  uint8_t* sDS = sP + kFaPBytes;                   // the dS tile, laid out like P
  float* sDelta = reinterpret_cast<float*>(sDS + kFaPBytes);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sDelta + kFaTile);
  uint64_t* v_full = bar + 0;
  uint64_t* v_empty = bar + 1;
  uint64_t* do_full = bar + 2;
  uint64_t* do_empty = bar + 3;
  uint64_t* q_full = bar + 4;
  uint64_t* q_empty = bar + 5;
  uint64_t* p_full = bar + 6;
  uint64_t* p_empty = bar + 7;
  uint64_t* dp_full = bar + 8;
  uint64_t* dp_empty = bar + 9;
  uint64_t* ds_full = bar + 10;
  uint64_t* ds_empty = bar + 11;
  uint64_t* acc_full = bar + 12;
  uint64_t* acc_empty = bar + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 14);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_t = (fp.L + kFaTile - 1) / kFaTile;   // query tiles = key tiles
  const int heads = fp.nh * fp.ns;
  const int num_items = n_t * heads;
  const uint32_t tile_tx = (uint32_t)fp.n_atoms * kFaAtomBytes;

  __shared__ int s_skip;
  if (threadIdx.x == 0) {
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    mbar_init(do_full, 1);
    mbar_init(do_empty, 1);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(p_full, 1);
    mbar_init(p_empty, 1 + kFbRowWarps);   // the products that read P, and the warps that read it
    mbar_init(dp_full, 1);
    mbar_init(dp_empty, kFbRowWarps);
    mbar_init(ds_full, kFbRowWarps);
    mbar_init(ds_empty, 1);
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kFbRowWarps);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mV);
    tma_prefetch_desc(&mQ);
    tma_prefetch_desc(&mdO);
    tma_prefetch_desc(&mP);
    tma_prefetch_desc(&mDelta);
    tma_prefetch_desc(&mDS);
    tma_prefetch_desc(&mdK);
    tma_prefetch_desc(&mdV);
  }
  if (warp == 1) {
    tmem_alloc<false>(tmem_slot, kFaTmemCols);
    tmem_relinquish<false>();
  }
  grid_dependency_wait();
  grid_launch_dependents();
  if (threadIdx.x == 0) s_skip = (status != nullptr && *reinterpret_cast<volatile int*>(status) != 0) ? 1 : 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int item_end = s_skip ? 0 : num_items;

  // item -> (key tile, head, sequence): the key tiles that see the most query tiles first
  auto decode = [&](int item, int& kt, int& hb, int& sb) {
    kt = item / heads;
    const int r = item % heads;
    hb = r % fp.nh;
    sb = r / fp.nh;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t nv = 0, ndo = 0, np = 0, nq = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < item_end && ok; item += gridDim.x) {
        int kt, hb, sb;
        decode(item, kt, hb, sb);
        if (!(ok = mbar_wait(v_empty, (nv & 1) ^ 1))) break;
        mbar_arrive_expect_tx(v_full, tile_tx);
        for (int a = 0; a < fp.n_atoms; ++a) tma_load_4d(sV + a * kFaAtomBytes, &mV, v_full, 64 * a, kt * kFaTile, hb, sb);
        ++nv;
        // in the order the MMA issuer frees them: dO_i and P_i, then Q_{i-1} (the
        // product dK += dS^T Q of a tile comes after dP and dV of the next one)
        auto load_q = [&](int i) -> bool {
          if (!mbar_wait(q_empty, (nq & 1) ^ 1)) return false;
          mbar_arrive_expect_tx(q_full, tile_tx);
          for (int a = 0; a < fp.n_atoms; ++a) tma_load_4d(sQ + a * kFaAtomBytes, &mQ, q_full, 64 * a, i * kFaTile, hb, sb);
          ++nq;
          return true;
        };
        for (int i = kt; i < n_t && ok; ++i) {
          if (!(ok = mbar_wait(do_empty, (ndo & 1) ^ 1))) break;
          mbar_arrive_expect_tx(do_full, tile_tx);
          for (int a = 0; a < fp.n_atoms; ++a)
            tma_load_4d(sdO + a * kFaAtomBytes, &mdO, do_full, 64 * a, i * kFaTile, hb, sb);
          ++ndo;
          if (!(ok = mbar_wait_cluster(p_empty, (np & 1) ^ 1))) break;
          mbar_arrive_expect_tx(p_full, kFaPBytes + kFaTile * sizeof(float));
          for (int a = 0; a < 2; ++a)
            tma_load_4d(sP + a * kFaAtomBytes, &mP, p_full, kt * kFaTile + 64 * a, i * kFaTile, hb, sb);
          tma_load_2d(sDelta, &mDelta, p_full, i * kFaTile, sb * fp.nh + hb, 0, false);
          ++np;
          if (i > kt) ok = load_q(i - 1);
        }
        if (ok) ok = load_q(n_t - 1);
      }
      if (!ok) record_status(status, kStatusTimeout, 30);
      // drain: every copy issued has landed before the CTA may exit
      if (nv > 0 && !mbar_wait(v_full, (nv - 1) & 1)) record_status(status, kStatusTimeout, 31);
      if (ndo > 0 && !mbar_wait(do_full, (ndo - 1) & 1)) record_status(status, kStatusTimeout, 31);
      if (np > 0 && !mbar_wait(p_full, (np - 1) & 1)) record_status(status, kStatusTimeout, 31);
      if (nq > 0 && !mbar_wait(q_full, (nq - 1) & 1)) record_status(status, kStatusTimeout, 31);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc_dp = make_idesc_bf16(kFaTile, kFaTile, false, false);
      const uint32_t idesc_dv = make_idesc_bf16(kFaTile, fp.d_pad, true, true);
      const uint32_t idesc_dk = make_idesc_bf16(kFaTile, fp.d_pad, true, true);
      const int nk_d = fp.d_pad / 16;
      const uint32_t t_dv = tmem_base, t_dk = tmem_base + 192u, t_dp = tmem_base + 384u;
      uint32_t nv = 0, ndo = 0, np = 0, nq = 0, ndp = 0, nds = 0, n_item = 0;
      bool ok = true;
      auto issue_dp = [&]() -> bool {  // dP = dO V^T (a query row per TMEM lane)
        if (!mbar_wait(do_full, ndo & 1) || !mbar_wait(dp_empty, (ndp & 1) ^ 1)) return false;
        tc_fence_after();
        const uint32_t vb = smem_u32(sV), ob = smem_u32(sdO);
        for (int kk = 0; kk < nk_d; ++kk) {
          const uint32_t off = (uint32_t)(kk >> 2) * kFaAtomBytes + (uint32_t)(kk & 3) * 32;
          umma_bf16(t_dp, make_sdesc_sw128(ob + off, 16, 1024), make_sdesc_sw128(vb + off, 16, 1024), idesc_dp,
                    kk > 0 ? 1u : 0u);
        }
        umma_commit(dp_full);
        ++ndp;
        return true;
      };
      auto issue_dv = [&](bool first) -> bool {  // dV += P^T dO
        if (!mbar_wait(p_full, np & 1)) return false;
        tc_fence_after();
        const uint32_t pb = smem_u32(sP), ob = smem_u32(sdO);
        for (int kk = 0; kk < kFaTile / 16; ++kk)
          umma_bf16(t_dv, make_sdesc_sw128(pb + kk * 2048, kFaAtomBytes, 1024),
                    make_sdesc_sw128(ob + kk * 2048, kFaAtomBytes, 1024), idesc_dv, (first && kk == 0) ? 0u : 1u);
        umma_commit(do_empty);
        umma_commit(p_empty);
        ++ndo;
        ++np;
        return true;
      };
      auto issue_dk = [&](bool first) -> bool {  // dK += dS^T Q (dS^T read as an MN-major operand)
        if (!mbar_wait(ds_full, nds & 1) || !mbar_wait(q_full, nq & 1)) return false;
        tc_fence_after();
        const uint32_t sb_ = smem_u32(sDS), qb = smem_u32(sQ);
        for (int kk = 0; kk < kFaTile / 16; ++kk)
          umma_bf16(t_dk, make_sdesc_sw128(sb_ + kk * 2048, kFaAtomBytes, 1024),
                    make_sdesc_sw128(qb + kk * 2048, kFaAtomBytes, 1024), idesc_dk, (first && kk == 0) ? 0u : 1u);
        umma_commit(q_empty);
        umma_commit(ds_empty);
        ++nq;
        ++nds;
        return true;
      };
      for (int item = blockIdx.x; item < item_end && ok; item += gridDim.x, ++n_item) {
        int kt, hb, sb;
        decode(item, kt, hb, sb);
        if (!(ok = mbar_wait(v_full, nv & 1))) break;
        ++nv;
        // the previous item's dK and dV have been read out of tensor memory
        if (!(ok = mbar_wait(acc_empty, (n_item & 1) ^ 1))) break;
        tc_fence_after();
        // dP and dV of query tile i, then dK of tile i - 1 (whose dS the threads have
        // been computing meanwhile)
        ok = issue_dp() && issue_dv(true);
        for (int i = kt + 1; i < n_t && ok; ++i) ok = issue_dp() && issue_dv(false) && issue_dk(i - 1 == kt);
        if (ok) ok = issue_dk(n_t - 1 == kt);
        if (ok) {
          umma_commit(v_empty);
          umma_commit(acc_full);
        }
      }
      if (!ok) record_status(status, kStatusTimeout, 32);
    }
  } else {
    // -------------------------------------------------------------- one query row per thread
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;                     // keys 64 half .. 64 half + 63 of each tile
    const int q_in = quarter * 32 + lane;                 // query row within the tile
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    uint32_t np = 0, ndp = 0, nds = 0, n_out = 0, n_item = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < item_end && ok; item += gridDim.x, ++n_item) {
      int kt, hb, sb;
      decode(item, kt, hb, sb);
      for (int i = kt; i < n_t && ok; ++i) {
        // dP row of query q_in of tile i, keys 0 .. 127 of tile kt
        if (!(ok = mbar_wait(dp_full, ndp & 1))) break;
        tc_fence_after();
        uint32_t dp[64];
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tmem_ld_32x32b_x32(t_lane + 384u + 64u * half + 32u * c, *reinterpret_cast<uint32_t(*)[32]>(&dp[32 * c]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dp_empty);
        ++ndp;
        // P (and delta) of tile (i, kt); the dS buffer free: dK's product read it,
        // and this warp's store of it has read it
        if (!(ok = mbar_wait(p_full, np & 1))) break;
        if (!(ok = mbar_wait(ds_empty, (nds & 1) ^ 1))) break;
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        const float dl = sDelta[q_in];
        const uint8_t* prow = sP + half * kFaAtomBytes + q_in * 128;
        uint8_t* dsrow = sDS + half * kFaAtomBytes + q_in * 128;
#pragma unroll
        for (int g = 0; g < 8; ++g) {           // keys 64 half + 8 g ..: chunk g ^ (q_in % 8) of atom `half`
          const uint32_t off = (uint32_t)((g ^ (q_in & 7)) << 4);
          const uint4 pv = *reinterpret_cast<const uint4*>(prow + off);
          const float pf[8] = {bf16lo(pv.x), bf16hi(pv.x), bf16lo(pv.y), bf16hi(pv.y),
                               bf16lo(pv.z), bf16hi(pv.z), bf16lo(pv.w), bf16hi(pv.w)};
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            pk[e] = pack_bf16x2(pf[2 * e] * (__uint_as_float(dp[8 * g + 2 * e]) - dl) * fp.alpha,
                                pf[2 * e + 1] * (__uint_as_float(dp[8 * g + 2 * e + 1]) - dl) * fp.alpha);
          *reinterpret_cast<uint4*>(dsrow + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(p_empty);
          tma_store_4d(&mDS, sDS + half * kFaAtomBytes + quarter * 32 * 128, kt * kFaTile + 64 * half,
                       i * kFaTile + quarter * 32, hb, sb);
          bulk_commit();
          mbar_arrive(ds_full);
        }
        ++np;
        ++nds;
      }
      if (!ok) break;
      // dS tile (query tile kt - 1, key tile kt) lies above the diagonal; the dQ
      // product of the 256-query tile that holds query tile kt - 1 reads it when kt
      // is odd, so it must hold zeros
      if (kt & 1) {
        for (int rr = half; rr < 32; rr += 4) {
          const int q = (kt - 1) * kFaTile + quarter * 32 + rr + 2 * (lane >> 4);
          const int c = kt * kFaTile + (lane & 15) * 8;
          if (c < fp.L) {
            uint16_t* row = fp.dS + (((int64_t)sb * fp.nh + hb) * fp.L + q) * (int64_t)fp.L;
            *reinterpret_cast<uint4*>(row + c) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      // dV and dK: bf16 through 32 x 32 boxes staged in this warp's own rows of the
      // dS buffer (its last store and dK's last product have read them)
      if (!(ok = mbar_wait(acc_full, n_item & 1))) break;
      tc_fence_after();
      if (lane == 0) bulk_wait_read<0>();
      __syncwarp();
      uint8_t* my_o = sDS + half * kFaAtomBytes + quarter * 32 * 128;   // 4 KB: two boxes
      for (int which = 0; which < 2; ++which) {
        const uint32_t col0 = which == 0 ? 0u : 192u;
        const CUtensorMap* map = which == 0 ? &mdV : &mdK;
        for (int c0 = 32 * half; c0 < fp.d_pad; c0 += 64) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_lane + col0 + (uint32_t)c0, r);
          tmem_ld_wait();
          if (c0 >= fp.d) continue;
          uint8_t* box = my_o + (n_out & 1) * kFaOStageBytes;
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint32_t off = lane * 64 + ((g ^ ((lane >> 1) & 3)) << 4);
            *reinterpret_cast<uint4*>(box + off) =
                make_uint4(pack_bf16x2(__uint_as_float(r[8 * g]), __uint_as_float(r[8 * g + 1])),
                           pack_bf16x2(__uint_as_float(r[8 * g + 2]), __uint_as_float(r[8 * g + 3])),
                           pack_bf16x2(__uint_as_float(r[8 * g + 4]), __uint_as_float(r[8 * g + 5])),
                           pack_bf16x2(__uint_as_float(r[8 * g + 6]), __uint_as_float(r[8 * g + 7])));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_4d(map, box, c0, kt * kFaTile + quarter * 32, hb, sb);
            bulk_commit();
          }
          ++n_out;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        bulk_wait_read<0>();   // the staged boxes have been read before the next dS rows land there
        mbar_arrive(acc_empty);
      }
    }
    if (!ok) record_status(status, kStatusTimeout, 33);
    if (lane == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<false>(tmem_base, kFaTmemCols);
  }
}

}  // namespace gbmlp

// Causal flash attention for head size 64 on the sm_103a tensor cores (tcgen05, TMEM,
// TMA).
//
// ujoy.net llm.c article, section "用C语言实现LLM": causal self-attention forward and
// backward.  Per head: S = Q K^T / sqrt(64) over keys j <= t, P = softmax(S), O = P V;
// the forward keeps O and each row's log-sum-exp only.
//
// Forward kernel, persistent, one CTA per SM, 320 threads; work item = (128-query
// tile, batch*head), heaviest tiles (most keys) first:
//   warp 0     TMA producer: Q tile (double-buffered across work items), then K and V
//              tiles of 128 keys through a 4-slot ring
//   warp 1     TMEM owner and MMA issuer: S = Q K^T (M=128, N=128, K=64) into one of two
//              TMEM S buffers, then O += P V (M=128, N=64, K=128) into the TMEM O buffer
//   warps 2-9  softmax, two warps per query row quadrant (each takes half the keys of a
//              tile): read the S row from TMEM, keep the running max / sum, write P
//              (bf16) into one of two shared buffers for the P V product; at the end
//              normalise O and write it with a TMA store, plus the row LSE
// The softmax reads its 64 scores of an S row from TMEM once (the S buffer is released
// right away, so S(j+2) can be computed while the softmax works on tile j), takes the
// row max over the warp pair, then the exponentials from registers.
// The exponent reference of a row (its max so far) is only raised when a new score
// exceeds it by more than 2^8: then, and only then, the row of O in TMEM is rescaled
// (after waiting for the P V in flight).  Numerator and denominator always use the same
// reference, so O / l is exact; p <= 256 stays far inside fp32 and bf16 range.  With P
// double-buffered, the softmax of tile j+1 never waits for P V of tile j, and S(j+1) is
// computed while the softmax works on tile j.  Every wait is bounded.
// The tensor maps are 3-D (columns, T, B) so no tile ever reads or writes past its own
// sequence.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "attention_tc.h"
#include "common.cuh"
#include "runtime.h"
#include "tc_ptx.cuh"
#include "../../include/gpt2.h"


#define AT_HS 64
#define AT_BM 128                  // queries per tile
#define AT_BN 128                  // keys per tile
#define AT_RING 4                  // K / V tile slots: K_{j+1} never waits on P V_{j-1}
#define AT_TILE_BYTES (128 * 64 * 2)
#define AT_THREADS 320               // producer, MMA issuer, 8 compute warps (2 per TMEM lane quadrant)
#define AT_LOG2E 1.4426950408889634f

#define AT_RESCALE_LOG2 8.0f        // raise a row's exponent reference only past 2^8

// 2^x with the hardware approximation (2 ulp); 2^-inf = 0.  P is rounded to bf16 and
// the row sum carries the same values, so the approximation cancels in O / l.
__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct AtSmem {
    static constexpr int Q_OFF = 0;                                          // 2 x 16 KB
    static constexpr int RING_OFF = Q_OFF + 2 * AT_TILE_BYTES;
    static constexpr int P_OFF = RING_OFF + AT_RING * AT_TILE_BYTES;         // 2 x (2 x 16 KB)
    static constexpr int O_OFF = P_OFF + 4 * AT_TILE_BYTES;                  // output staging
    static constexpr int X_OFF = O_OFF + AT_TILE_BYTES;                      // row max / sum exchange
    static constexpr int BAR_OFF = X_OFF + 3 * 1024;
    // q_full[2], q_empty[2], ring_full[4], ring_empty[4], s_full[2], s_free[2],
    // p_full[2], o_done[2], o_free, done; then tmem address and abort flag
    static constexpr int NBAR = 4 + 2 * AT_RING + 4 + 4 + 2;
    static constexpr int TOTAL = BAR_OFF + NBAR * 8 + 16 + 1024;
};

__global__ void __launch_bounds__(AT_THREADS, 1)
attention_tc_forward_kernel(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmO,
                            float* __restrict__ lse, int B, int Tn, int C, int NH, unsigned* err) {
    using S = AtSmem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
    uint64_t* q_full = bars;
    uint64_t* q_empty = bars + 2;
    uint64_t* ring_full = bars + 4;
    uint64_t* ring_empty = ring_full + AT_RING;
    uint64_t* s_full = ring_empty + AT_RING;
    uint64_t* s_free = s_full + 2;
    uint64_t* p_full = s_free + 2;
    uint64_t* o_done = p_full + 2;
    uint64_t* o_free = o_done + 2;
    uint64_t* done = o_free + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = B * NH;
    const int nqt = (Tn + AT_BM - 1) / AT_BM;
    const int n_items = nqt * BH;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) { mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1); }
        for (int i = 0; i < AT_RING; i++) { mbar_init(&ring_full[i], 1); mbar_init(&ring_empty[i], 1); }
        for (int i = 0; i < 2; i++) { mbar_init(&s_full[i], 1); mbar_init(&s_free[i], 8); }
        for (int i = 0; i < 2; i++) { mbar_init(&p_full[i], 8); mbar_init(&o_done[i], 1); }
        mbar_init(o_free, 8);
        mbar_init(done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tmQKV);
        tma_prefetch_desc(&tmO);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(512) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t TM_S = tmem_base;          // S buffers at columns 0 and 128
    const uint32_t TM_O = tmem_base + 256;    // O at columns 256..319

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int rc = 0, local = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, local++) {
                const int qt = nqt - 1 - it / BH, bh = it % BH, b = bh / NH, h = bh % NH;
                const int qb = local & 1;
                if (!mbar_wait(&q_empty[qb], ((local >> 1) & 1) ^ 1, abort_flag, err)) break;
                mbar_expect_tx(&q_full[qb], AT_TILE_BYTES);
                tma_load_3d(smem + S::Q_OFF + qb * AT_TILE_BYTES, &tmQKV, &q_full[qb], h * AT_HS, qt * AT_BM, b);
                const int nk = qt + 1;
                for (int j = 0; j < nk && ok; j++) {
                    for (int kv = 0; kv < 2; kv++, rc++) {
                        const int s = rc % AT_RING;
                        if (!mbar_wait(&ring_empty[s], ((rc / AT_RING) & 1) ^ 1, abort_flag, err)) { ok = false; break; }
                        mbar_expect_tx(&ring_full[s], AT_TILE_BYTES);
                        tma_load_3d(smem + S::RING_OFF + s * AT_TILE_BYTES, &tmQKV, &ring_full[s],
                                    (kv + 1) * C + h * AT_HS, j * AT_BN, b);
                    }
                }
            }
            // in-flight copies land before the CTA retires
            for (int back = 0; back < AT_RING && back < rc; back++) {
                const int k = rc - 1 - back;
                const long long t0 = clock64();
                while (!mbar_try_wait(&ring_full[k % AT_RING], (k / AT_RING) & 1))
                    if (clock64() - t0 > TC_WAIT_LIMIT) { raise_error(err, ERRBIT_TIMEOUT); break; }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(AT_BM, AT_BN, false, false);
            constexpr uint32_t IDESC_O = idesc_bf16(AT_BM, AT_HS, false, true);
            int rc = 0, sc = 0, pc = 0, local = 0;
            bool ok = true;
            // S = Q K^T for the K tile at ring index kidx into S buffer sc % 2
            auto issue_s = [&](uint32_t q_addr, int kidx) -> bool {
                const int sb = sc & 1, slot = kidx % AT_RING;
                if (!mbar_wait(&s_free[sb], ((sc >> 1) & 1) ^ 1, abort_flag, err)) return false;
                if (!mbar_wait(&ring_full[slot], (kidx / AT_RING) & 1, abort_flag, err)) return false;
                tc_fence_after();
                const uint32_t k_addr = smem_u32(smem + S::RING_OFF + slot * AT_TILE_BYTES);
#pragma unroll
                for (int k = 0; k < AT_HS / 16; k++)
                    tc_mma(TM_S + sb * AT_BN, sdesc(q_addr + k * 32, 16, 1024), sdesc(k_addr + k * 32, 16, 1024),
                           IDESC_S, k > 0 ? 1u : 0u);
                tc_commit(&s_full[sb]);
                tc_commit(&ring_empty[slot]);
                sc++;
                return true;
            };
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, local++) {
                const int qt = nqt - 1 - it / BH;
                const int nk = qt + 1;
                const int qb = local & 1;
                if (!mbar_wait(&q_full[qb], (local >> 1) & 1, abort_flag, err)) break;
                const uint32_t q_addr = smem_u32(smem + S::Q_OFF + qb * AT_TILE_BYTES);
                // K_j sits at ring index rc + 2j, V_j at rc + 2j + 1
                if (!issue_s(q_addr, rc)) break;
                for (int j = 0; j < nk && ok; j++) {
                    if (j + 1 < nk && !issue_s(q_addr, rc + 2 * (j + 1))) { ok = false; break; }
                    if (j == nk - 1) tc_commit(&q_empty[qb]);   // Q buffer free once the last S completes
                    // O += P_j V_j, P_j in buffer pc % 2
                    const int vidx = rc + 2 * j + 1, vslot = vidx % AT_RING;
                    const int pb = pc & 1;
                    if (!mbar_wait(&ring_full[vslot], (vidx / AT_RING) & 1, abort_flag, err)) { ok = false; break; }
                    if (!mbar_wait(&p_full[pb], (pc >> 1) & 1, abort_flag, err)) { ok = false; break; }
                    if (j == 0 && local > 0 && !mbar_wait(o_free, (local - 1) & 1, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t p_addr = smem_u32(smem + S::P_OFF + pb * 2 * AT_TILE_BYTES);
                    const uint32_t v_addr = smem_u32(smem + S::RING_OFF + vslot * AT_TILE_BYTES);
#pragma unroll
                    for (int k = 0; k < AT_BN / 16; k++)
                        tc_mma(TM_O, sdesc(p_addr + (k >> 2) * AT_TILE_BYTES + (k & 3) * 32, 16, 1024),
                               sdesc(v_addr + k * 2048, 8192, 1024), IDESC_O, (j > 0 || k > 0) ? 1u : 0u);
                    tc_commit(&o_done[pb]);
                    tc_commit(&ring_empty[vslot]);
                    pc++;
                }
                rc += 2 * nk;
            }
            tc_commit(done);
            const long long t0 = clock64();
            while (!mbar_try_wait(done, 0))
                if (clock64() - t0 > TC_WAIT_LIMIT) { raise_error(err, ERRBIT_TIMEOUT); break; }
        }
    } else {
        // ------------------------------------------------------------ softmax warps 2..9
        // Two warps per TMEM lane quadrant: `half` picks columns [64*half, 64*half + 64) of
        // every S tile (and [32*half, 32*half + 32) of O).  The pair swaps its row maxima
        // through shared memory once per tile; the row sums stay split until the end.
        const int lane_grp = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = lane_grp * 32 + lane;                 // query row in the tile
        const uint32_t lrow = (uint32_t)(lane_grp * 32) << 16;
        uint8_t* obuf = smem + S::O_OFF;
        float* xmax = reinterpret_cast<float*>(smem + S::X_OFF);   // [tile parity][half][128]
        float* xsum = xmax + 512;                                   // [half][128]
        const int pair_bar = 2 + lane_grp;                          // named barrier of the pair
        const float sl2 = AT_LOG2E * 0.125f;                // log2(e) / sqrt(64)
        int sc = 0, pc = 0, local = 0;
        int seen0 = 0, seen1 = 0;                           // o_done phases observed, per P buffer
        bool alive = true;
        // wait until P V number `i` has completed (phases of each buffer are observed in order)
        auto wait_pv = [&](int i) -> bool {
            const int bb = i & 1, ph = i >> 1;
            if ((bb ? seen1 : seen0) > ph) return true;
            int okw = 1;
            if (lane == 0) okw = mbar_wait(&o_done[bb], ph & 1, abort_flag, err) ? 1 : 0;
            okw = __shfl_sync(0xffffffffu, okw, 0);
            if (bb) seen1 = ph + 1; else seen0 = ph + 1;
            __syncwarp();
            return okw != 0;
        };
        for (int it = blockIdx.x; it < n_items && alive; it += gridDim.x, local++) {
            const int qt = nqt - 1 - it / BH, bh = it % BH, b = bh / NH, h = bh % NH;
            const int nk = qt + 1;
            const int q = qt * AT_BM + r;
            const int pc0 = pc;                             // index of this item's first P V
            float m = -INFINITY, l = 0.f;                   // exponent reference, partial running sum
            for (int j = 0; j < nk; j++) {
                const int sb = sc & 1;
                int okw = 1;
                if (lane == 0) okw = mbar_wait(&s_full[sb], (sc >> 1) & 1, abort_flag, err) ? 1 : 0;
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (!okw) { alive = false; break; }
                __syncwarp();
                tc_fence_after();
                const uint32_t srow = TM_S + sb * AT_BN + lrow;
                // keys after the query are masked on the diagonal tile: columns > lim
                const int lim = (j == nk - 1) ? (q - j * AT_BN) : AT_BN;
                const bool masked = lim < AT_BN;            // only the diagonal tile
                // this warp's 64 scores of the row, read once; the S buffer is then free
                uint32_t sr[64];
                {
                    uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
                    uint32_t (&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
                    tmem_ld32(srow + half * 64, s0);
                    tmem_ld32(srow + half * 64 + 32, s1);
                    tmem_ld_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[sb]);
                if (masked) {
#pragma unroll
                    for (int i = 0; i < 64; i++)
                        if (half * 64 + i > lim) sr[i] = __float_as_uint(-INFINITY);
                }
                // max over this warp's 64 columns, then over the pair
                float mx;
                {
                    // 64 -> 22 -> 8 -> 3 -> 1 with three-input maxima
                    float a[22], b[8];
#pragma unroll
                    for (int i = 0; i < 21; i++)
                        a[i] = fmax3(__uint_as_float(sr[3 * i]), __uint_as_float(sr[3 * i + 1]), __uint_as_float(sr[3 * i + 2]));
                    a[21] = __uint_as_float(sr[63]);
#pragma unroll
                    for (int i = 0; i < 7; i++) b[i] = fmax3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
                    b[7] = a[21];
                    mx = fmax3(fmax3(b[0], b[1], b[2]), fmax3(b[3], b[4], b[5]), fmaxf(b[6], b[7]));
                }
                mx *= sl2;                                  // scaling by sl2 > 0 keeps the max
                float* xm = xmax + (sc & 1) * 256;
                xm[half * 128 + r] = mx;
                named_bar(pair_bar, 64);
                mx = fmaxf(mx, xm[(half ^ 1) * 128 + r]);
                // raise the reference only when needed; then O must be rescaled, after the
                // P V still in flight for this item has landed
                const bool raise = mx > m + AT_RESCALE_LOG2;
                const float m_new = raise ? mx : m;
                const float corr = ex2_fast(m - m_new);     // 1 when unchanged, 0 on the first tile
                if (__any_sync(0xffffffffu, raise && j > 0)) {
                    if (!wait_pv(pc0 + j - 1)) { alive = false; break; }
                    tc_fence_after();
                    uint32_t rr[32];
                    tmem_ld32(TM_O + lrow + half * 32, rr);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i++) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * corr);
                    tmem_st32(TM_O + lrow + half * 32, rr);
                    tmem_st_wait();
                }
                m = m_new;
                // the P buffer of this tile was last read by P V two tiles back
                const int pb = pc & 1;
                if (pc >= 2 && !wait_pv(pc - 2)) { alive = false; break; }
                uint8_t* pbuf = smem + S::P_OFF + pb * 2 * AT_TILE_BYTES;
                // p = 2^(s - m) (masked scores are -inf: p = 0), partial row sum, P into the
                // swizzled A operand
                float rs = 0.f;
#pragma unroll
                for (int h2 = 0; h2 < 2; h2++) {
                    const int c = half * 64 + h2 * 32;
                    float p[32];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float2 a = __ffma2_rn(make_float2(__uint_as_float(sr[h2 * 32 + i]), __uint_as_float(sr[h2 * 32 + i + 1])),
                                                    make_float2(sl2, sl2), make_float2(-m, -m));
                        p[i] = ex2_fast(a.x);
                        p[i + 1] = ex2_fast(a.y);
                    }
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        const int ch = (c >> 3) + k;
                        Vec<bf16> pv;
#pragma unroll
                        for (int e = 0; e < 8; e += 2) pv.set2(e, p[8 * k + e], p[8 * k + e + 1]);
                        *reinterpret_cast<uint4*>(pbuf + (ch >> 3) * AT_TILE_BYTES + r * 128 +
                                                  (((ch & 7) ^ (r & 7)) << 4)) = pv.v;
                    }
                    // pairwise tree sum; the levels with w >= 2 in packed pairs
#pragma unroll
                    for (int w = 16; w > 1; w >>= 1)
#pragma unroll
                        for (int i = 0; i < w; i += 2) {
                            const float2 x = __fadd2_rn(make_float2(p[i], p[i + 1]), make_float2(p[i + w], p[i + w + 1]));
                            p[i] = x.x;
                            p[i + 1] = x.y;
                        }
                    rs += p[0] + p[1];
                }
                l = l * corr + rs;
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[pb]);
                sc++;
                pc++;
            }
            if (!alive) break;
            // the last P V of the item, then normalise and write this row of O
            if (!wait_pv(pc - 1)) break;
            tc_fence_after();
            float o[32];
            {
                uint32_t rr[32];
                tmem_ld32(TM_O + lrow + half * 32, rr);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; i++) o[i] = __uint_as_float(rr[i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
            xsum[half * 128 + r] = l;
            named_bar(pair_bar, 64);
            const float lt = l + xsum[(half ^ 1) * 128 + r];
            const float inv = 1.0f / lt;
            // the previous item's O store must have finished reading the staging buffer
            if (threadIdx.x == 64) bulk_wait_read<0>();
            named_bar(1, 256);
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const int ch = half * 4 + k;
                Vec<bf16> ov;
#pragma unroll
                for (int e = 0; e < 8; e += 2) ov.set2(e, o[8 * k + e] * inv, o[8 * k + e + 1] * inv);
                *reinterpret_cast<uint4*>(obuf + r * 128 + ((ch ^ (r & 7)) << 4)) = ov.v;
            }
            fence_async_smem();
            named_bar(1, 256);
            if (threadIdx.x == 64) {
                tma_store_3d(&tmO, obuf, h * AT_HS, qt * AT_BM, b);
                bulk_commit();
            }
            if (half == 0 && q < Tn) lse[(size_t)bh * Tn + q] = (m + log2f(lt)) / AT_LOG2E;
        }
        if (threadIdx.x == 64) bulk_wait<0>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    __syncwarp();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512) : "memory");
}

// ==================================================================== backward
// One kernel, two modes (no atomics, deterministic):
//   DKV  item = (128-key tile t, b*h); for every query tile u >= t:
//          S^T = K_t Q_u^T, dP^T = V_t dO_u^T                 (TMEM, M=128 N=128 K=64)
//          P^T = 2^(S^T log2e/8 - LSE_u log2e), dS^T = P^T (dP^T - D_u)   (compute warps)
//          dV += P^T dO_u, dK += dS^T Q_u                     (TMEM, M=128 N=64 K=128)
//        then dK / 8 and dV go to dqkv by TMA store.
//   DQ   item = (128-query tile t, b*h); for every key tile u <= t:
//          S = Q_t K_u^T, dP = dO_t V_u^T; P = 2^(S log2e/8 - LSE log2e), dS = P (dP - D)
//          dQ += dS K_u;  then dQ / 8 to dqkv.
// Warp 0 loads (the item's two row tiles once; the per-u tiles through a 3-stage ring
// with, in DKV mode, that u's LSE and D vectors); warp 1 issues
// the MMAs (the next S/dP pair is issued before the dV/dK (dQ) products of the current
// one); warps 2-9 compute, two warps per TMEM lane quadrant, each on half the columns of
// a tile (a TMEM lane is a key row in DKV mode, a query row in DQ mode).  The operands
// the compute warps produce for the products are double-buffered, so tile u+1 is
// computed while the products of tile u run: dS (dS^T) in shared memory and, in DKV
// mode, P^T (bf16, two per 32-bit column) in TMEM, read there as the A operand of
// dV += P^T dO_u.
#define AB_STAGE_BYTES (2 * AT_TILE_BYTES + 1024)   // two tiles + LSE[128] + D[128]

template <bool DKV>
struct AbSmem {
    static constexpr int RING = 3;
    static constexpr int R_OFF = 0;                                        // 2 row tiles
    static constexpr int RING_OFF = R_OFF + 2 * AT_TILE_BYTES;
    static constexpr int DS_OFF = RING_OFF + RING * AB_STAGE_BYTES;        // 2 x dS or dS^T, 32 KB each
    static constexpr int BAR_OFF = DS_OFF + 4 * AT_TILE_BYTES;
    // rr_full, rr_empty, ring_full[RING], ring_empty[RING], x_full, x_free, pds_full[2],
    // pds_free[2], acc_free, done; tmem address, abort flag
    static constexpr int NBAR = 2 + 2 * RING + 8;
    static constexpr int TOTAL = BAR_OFF + NBAR * 8 + 16 + 1024;
};

template <bool DKV>
__global__ void __launch_bounds__(AT_THREADS, 1)
attention_tc_backward_kernel(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmDO,
                             const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmD,
                             const __grid_constant__ CUtensorMap tmDQKV, const float* __restrict__ lse,
                             const float* __restrict__ Dsum, int B, int Tn, int Tp, int C, int NH, unsigned* err) {
    using S = AbSmem<DKV>;
    constexpr int AB_RING = S::RING;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
    uint64_t* rr_full = bars;
    uint64_t* rr_empty = bars + 1;
    uint64_t* ring_full = bars + 2;
    uint64_t* ring_empty = ring_full + AB_RING;
    uint64_t* x_full = ring_empty + AB_RING;
    uint64_t* x_free = x_full + 1;
    uint64_t* pds_full = x_free + 1;       // [2]
    uint64_t* pds_free = pds_full + 2;     // [2]
    uint64_t* acc_free = pds_free + 2;
    uint64_t* done = acc_free + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = B * NH;
    const int nt = (Tn + AT_BM - 1) / AT_BM;
    const int n_items = nt * BH;
    // item -> (row tile, bh, range of u), heaviest items first
    auto item_of = [&](int it, int& t, int& bh, int& u0, int& u1) {
        bh = it % BH;
        if (DKV) { t = it / BH; u0 = t; u1 = nt; }
        else { t = nt - 1 - it / BH; u0 = 0; u1 = t + 1; }
    };

    if (threadIdx.x == 0) {
        mbar_init(rr_full, 1);
        mbar_init(rr_empty, 1);
        for (int i = 0; i < AB_RING; i++) { mbar_init(&ring_full[i], 1); mbar_init(&ring_empty[i], 1); }
        mbar_init(x_full, 1);
        mbar_init(x_free, 8);
        for (int i = 0; i < 2; i++) { mbar_init(&pds_full[i], 8); mbar_init(&pds_free[i], 1); }
        mbar_init(acc_free, 8);
        mbar_init(done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tmQKV);
        tma_prefetch_desc(&tmDO);
        tma_prefetch_desc(&tmDQKV);
        if (DKV) { tma_prefetch_desc(&tmL); tma_prefetch_desc(&tmD); }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(512) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // S (S^T), dP (dP^T), dV or dQ, dK, then (DKV) two P^T buffers of 64 columns
    const uint32_t TM_X1 = tmem_base, TM_X2 = tmem_base + 128, TM_A1 = tmem_base + 256, TM_A2 = tmem_base + 320;
    const uint32_t TM_P = tmem_base + 384;

    if (warp == 0) {
        // ------------------------------------------------------------ loads
        if (lane == 0) {
            int rc = 0, local = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, local++) {
                int t, bh, u0, u1;
                item_of(it, t, bh, u0, u1);
                const int b = bh / NH, h = bh % NH;
                if (!mbar_wait(rr_empty, (local & 1) ^ 1, abort_flag, err)) break;
                mbar_expect_tx(rr_full, 2 * AT_TILE_BYTES);
                if (DKV) {
                    tma_load_3d(smem + S::R_OFF, &tmQKV, rr_full, C + h * AT_HS, t * AT_BM, b);                  // K_t
                    tma_load_3d(smem + S::R_OFF + AT_TILE_BYTES, &tmQKV, rr_full, 2 * C + h * AT_HS, t * AT_BM, b);  // V_t
                } else {
                    tma_load_3d(smem + S::R_OFF, &tmQKV, rr_full, h * AT_HS, t * AT_BM, b);                      // Q_t
                    tma_load_3d(smem + S::R_OFF + AT_TILE_BYTES, &tmDO, rr_full, h * AT_HS, t * AT_BM, b);       // dO_t
                }
                for (int u = u0; u < u1; u++, rc++) {
                    const int slot = rc % AB_RING;
                    if (!mbar_wait(&ring_empty[slot], ((rc / AB_RING) & 1) ^ 1, abort_flag, err)) { ok = false; break; }
                    uint8_t* st = smem + S::RING_OFF + slot * AB_STAGE_BYTES;
                    if (DKV) {
                        mbar_expect_tx(&ring_full[slot], 2 * AT_TILE_BYTES + 1024);
                        tma_load_3d(st, &tmQKV, &ring_full[slot], h * AT_HS, u * AT_BM, b);                       // Q_u
                        tma_load_3d(st + AT_TILE_BYTES, &tmDO, &ring_full[slot], h * AT_HS, u * AT_BM, b);        // dO_u
                        tma_load_2d(st + 2 * AT_TILE_BYTES, &tmL, &ring_full[slot], u * AT_BM, bh);               // LSE_u
                        tma_load_2d(st + 2 * AT_TILE_BYTES + 512, &tmD, &ring_full[slot], u * AT_BM, bh);         // D_u
                    } else {
                        mbar_expect_tx(&ring_full[slot], 2 * AT_TILE_BYTES);
                        tma_load_3d(st, &tmQKV, &ring_full[slot], C + h * AT_HS, u * AT_BM, b);                   // K_u
                        tma_load_3d(st + AT_TILE_BYTES, &tmQKV, &ring_full[slot], 2 * C + h * AT_HS, u * AT_BM, b);  // V_u
                    }
                }
            }
            for (int back = 0; back < AB_RING && back < rc; back++) {
                const int k = rc - 1 - back;
                const long long t0 = clock64();
                while (!mbar_try_wait(&ring_full[k % AB_RING], (k / AB_RING) & 1))
                    if (clock64() - t0 > TC_WAIT_LIMIT) { raise_error(err, ERRBIT_TIMEOUT); break; }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_X = idesc_bf16(AT_BM, AT_BN, false, false);
            constexpr uint32_t IDESC_A = idesc_bf16(AT_BM, AT_HS, false, true);
            const uint32_t r0 = smem_u32(smem + S::R_OFF), r1 = r0 + AT_TILE_BYTES;
            const uint32_t dsbase = smem_u32(smem + S::DS_OFF);
            int rc = 0, xc = 0, gc = 0, local = 0;
            bool ok = true;
            // the S / dP pair for the ring stage of index `idx`
            auto issue_x = [&](int idx) -> bool {
                const int slot = idx % AB_RING;
                if (!mbar_wait(&ring_full[slot], (idx / AB_RING) & 1, abort_flag, err)) return false;
                if (!mbar_wait(x_free, (xc & 1) ^ 1, abort_flag, err)) return false;
                tc_fence_after();
                const uint32_t st = smem_u32(smem + S::RING_OFF + slot * AB_STAGE_BYTES);
#pragma unroll
                for (int k = 0; k < AT_HS / 16; k++)
                    tc_mma(TM_X1, sdesc(r0 + k * 32, 16, 1024), sdesc(st + k * 32, 16, 1024), IDESC_X, k > 0);
#pragma unroll
                for (int k = 0; k < AT_HS / 16; k++)
                    tc_mma(TM_X2, sdesc(r1 + k * 32, 16, 1024), sdesc(st + AT_TILE_BYTES + k * 32, 16, 1024), IDESC_X,
                           k > 0);
                tc_commit(x_full);
                xc++;
                return true;
            };
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, local++) {
                int t, bh, u0, u1;
                item_of(it, t, bh, u0, u1);
                const int nu = u1 - u0;
                if (!mbar_wait(rr_full, local & 1, abort_flag, err)) break;
                if (!issue_x(rc)) break;
                for (int i = 0; i < nu && ok; i++) {
                    if (i + 1 < nu && !issue_x(rc + i + 1)) { ok = false; break; }
                    if (i == nu - 1) tc_commit(rr_empty);          // row tiles free after the last S / dP
                    const int slot = (rc + i) % AB_RING;
                    const uint32_t st = smem_u32(smem + S::RING_OFF + slot * AB_STAGE_BYTES);
                    const int pb = gc & 1;                           // P / dS buffer of this tile
                    const uint32_t dsbuf = dsbase + pb * 2 * AT_TILE_BYTES;
                    if (!mbar_wait(&pds_full[pb], (gc >> 1) & 1, abort_flag, err)) { ok = false; break; }
                    if (i == 0 && local > 0 && !mbar_wait(acc_free, (local - 1) & 1, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    if (DKV) {
                        // dV += P^T dO_u (P^T from TMEM, 8 columns per 16 queries) ; dK += dS^T Q_u
                        const uint32_t pt = TM_P + pb * 64;
#pragma unroll
                        for (int k = 0; k < AT_BN / 16; k++) {
                            const uint32_t aoff = (k >> 2) * AT_TILE_BYTES + (k & 3) * 32;
                            tc_mma_ts(TM_A1, pt + k * 8, sdesc(st + AT_TILE_BYTES + k * 2048, 8192, 1024), IDESC_A,
                                      (i > 0 || k > 0));
                            tc_mma(TM_A2, sdesc(dsbuf + aoff, 16, 1024), sdesc(st + k * 2048, 8192, 1024), IDESC_A,
                                   (i > 0 || k > 0));
                        }
                    } else {
                        // dQ += dS K_u
#pragma unroll
                        for (int k = 0; k < AT_BN / 16; k++)
                            tc_mma(TM_A1, sdesc(dsbuf + (k >> 2) * AT_TILE_BYTES + (k & 3) * 32, 16, 1024),
                                   sdesc(st + k * 2048, 8192, 1024), IDESC_A, (i > 0 || k > 0));
                    }
                    tc_commit(&pds_free[pb]);
                    tc_commit(&ring_empty[slot]);
                    gc++;
                }
                rc += nu;
            }
            tc_commit(done);
            const long long t0 = clock64();
            while (!mbar_try_wait(done, 0))
                if (clock64() - t0 > TC_WAIT_LIMIT) { raise_error(err, ERRBIT_TIMEOUT); break; }
        }
    } else {
        // ------------------------------------------------------------ compute warps 2..9
        const int lane_grp = warp & 3;
        const int half = (warp - 2) >> 2;                   // columns [64*half, 64*half + 64) of a tile
        const int r = lane_grp * 32 + lane;                 // TMEM lane = row of the item's tile
        const uint32_t lrow = (uint32_t)(lane_grp * 32) << 16;
        const float sl2 = AT_LOG2E * 0.125f;
        uint8_t* dsbase = smem + S::DS_OFF;
        int rc = 0, xc = 0, gc = 0, local = 0;
        int pf_seen0 = 0, pf_seen1 = 0;                     // pds_free completions observed per buffer
        int stg_pending = -1;                               // dS buffer an item's store may still be reading
        // before this buffer is written again, the store issued from it has read it
        auto stg_release = [&](int buf) {
            if (stg_pending != buf) return;
            if (threadIdx.x == 64) bulk_wait_read<0>();
            named_bar(1, 256);
            stg_pending = -1;
        };
        bool alive = true;
        auto wait_one = [&](uint64_t* bar, uint32_t parity) -> bool {
            int okw = 1;
            if (lane == 0) okw = mbar_wait(bar, parity, abort_flag, err) ? 1 : 0;
            okw = __shfl_sync(0xffffffffu, okw, 0);
            __syncwarp();
            return okw != 0;
        };
        // wait for the dV/dK (dQ) products of tile n: completion n >> 1 of buffer n & 1's
        // barrier (each buffer's completions are observed in order)
        auto wait_pds_free = [&](int n) -> bool {
            const int b = n & 1, need = (n >> 1) + 1;
            if (b == 0) {
                if (pf_seen0 >= need) return true;
                pf_seen0 = need;
            } else {
                if (pf_seen1 >= need) return true;
                pf_seen1 = need;
            }
            return wait_one(&pds_free[b], (n >> 1) & 1);
        };
        for (int it = blockIdx.x; it < n_items && alive; it += gridDim.x, local++) {
            int t, bh, u0, u1;
            item_of(it, t, bh, u0, u1);
            const int b = bh / NH, h = bh % NH;
            const int grow = t * AT_BM + r;                 // this thread's key (DKV) or query (DQ)
            float Lrow = 0.f, Drow = 0.f;
            if (!DKV && grow < Tn) {
                Lrow = lse[(size_t)bh * Tp + grow] * AT_LOG2E;
                Drow = Dsum[(size_t)bh * Tp + grow];
            }
            for (int u = u0; u < u1; u++, rc++, xc++, gc++) {
                if (!wait_one(x_full, xc & 1)) { alive = false; break; }
                tc_fence_after();
                const uint8_t* st = smem + S::RING_OFF + (rc % AB_RING) * AB_STAGE_BYTES;
                const float* Lv = reinterpret_cast<const float*>(st + 2 * AT_TILE_BYTES);
                const float* Dv = Lv + 128;
                const int pb = gc & 1;
                uint8_t* dsbuf = dsbase + pb * 2 * AT_TILE_BYTES;
#pragma unroll 1
                for (int c = half * 64; c < half * 64 + 64; c += 32) {
                    uint32_t s1[32], s2[32];
                    tmem_ld32(TM_X1 + lrow + c, s1);
                    tmem_ld32(TM_X2 + lrow + c, s2);
                    tmem_ld_wait();
                    if (c == half * 64 + 32) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(x_free);      // S / dP TMEM may be overwritten
                    }
                    float p[32], ds[32];
                    float Lc[32], Dc[32];
                    if (DKV) {
                        // LSE (to the exp2 domain) and D of these 32 query columns
#pragma unroll
                        for (int k = 0; k < 8; k++) {
                            const float4 lv = *reinterpret_cast<const float4*>(Lv + c + 4 * k);
                            const float4 dv = *reinterpret_cast<const float4*>(Dv + c + 4 * k);
                            Lc[4 * k] = lv.x * AT_LOG2E; Lc[4 * k + 1] = lv.y * AT_LOG2E;
                            Lc[4 * k + 2] = lv.z * AT_LOG2E; Lc[4 * k + 3] = lv.w * AT_LOG2E;
                            Dc[4 * k] = dv.x; Dc[4 * k + 1] = dv.y; Dc[4 * k + 2] = dv.z; Dc[4 * k + 3] = dv.w;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i++) { Lc[i] = Lrow; Dc[i] = Drow; }
                    }
                    // masking is needed only where the tile meets the diagonal or the end of T
                    const int col0 = u * AT_BN + c;
                    const bool masked = DKV ? (col0 < grow + 1 || col0 + 31 >= Tn) : (col0 + 31 > grow);
                    if (masked) {
#pragma unroll
                        for (int i = 0; i < 32; i++) {
                            const int col = col0 + i;            // query (DKV) or key (DQ) index
                            const bool valid = DKV ? ((col >= grow) && (col < Tn)) : (col <= grow);
                            const float pv = ex2_fast(fmaf(__uint_as_float(s1[i]), sl2, -Lc[i]));
                            p[i] = valid ? pv : 0.f;
                            ds[i] = valid ? pv * (__uint_as_float(s2[i]) - Dc[i]) : 0.f;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 a = __ffma2_rn(make_float2(__uint_as_float(s1[i]), __uint_as_float(s1[i + 1])),
                                                        make_float2(sl2, sl2), make_float2(-Lc[i], -Lc[i + 1]));
                            p[i] = ex2_fast(a.x);
                            p[i + 1] = ex2_fast(a.y);
                            const float2 d = __fadd2_rn(make_float2(__uint_as_float(s2[i]), __uint_as_float(s2[i + 1])),
                                                        make_float2(-Dc[i], -Dc[i + 1]));
                            const float2 g = __fmul2_rn(make_float2(p[i], p[i + 1]), d);
                            ds[i] = g.x;
                            ds[i + 1] = g.y;
                        }
                    }
                    // the products of tile gc-2, and an item's output store, must have
                    // finished reading this buffer
                    if (c == half * 64 && gc >= 2 && !wait_pds_free(gc - 2)) { alive = false; break; }
                    if (c == half * 64) stg_release(pb);
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        const int ch = (c >> 3) + k;
                        const int off = (ch >> 3) * AT_TILE_BYTES + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
                        Vec<bf16> dv;
#pragma unroll
                        for (int e = 0; e < 8; e += 2) dv.set2(e, ds[8 * k + e], ds[8 * k + e + 1]);
                        *reinterpret_cast<uint4*>(dsbuf + off) = dv.v;
                    }
                    if (DKV) {
                        // P^T row r, queries c..c+31: 16 columns of bf16 pairs
                        uint32_t pk[16];
#pragma unroll
                        for (int k = 0; k < 16; k++) {
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(p[2 * k], p[2 * k + 1]);
                            pk[k] = *reinterpret_cast<uint32_t*>(&h2);
                        }
                        tmem_st16(TM_P + pb * 64 + lrow + (c >> 1), pk);
                    }
                }
                if (!alive) break;
                if (DKV) tmem_st_wait();
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&pds_full[pb]);
            }
            if (!alive) break;
            // accumulators of the item: wait for its last products, read, release, store
            if (!wait_pds_free(gc - 1)) break;
            // staging: the last tile's dS buffer (its products are done; the next item's
            // first tile uses the other buffer)
            uint8_t* stg = dsbase + ((gc - 1) & 1) * 2 * AT_TILE_BYTES;
            stg_release((gc - 1) & 1);
            tc_fence_after();
            float a1[32], a2[32];
            {
                uint32_t rr[32];
                tmem_ld32(TM_A1 + lrow + half * 32, rr);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; i++) a1[i] = __uint_as_float(rr[i]);
                if (DKV) {
                    tmem_ld32(TM_A2 + lrow + half * 32, rr);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i++) a2[i] = __uint_as_float(rr[i]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free);
            // stage in the (now idle) P / dS buffers, 128B-swizzled rows, then TMA-store
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const int ch = half * 4 + k;
                const int off = r * 128 + ((ch ^ (r & 7)) << 4);
                Vec<bf16> v1;
                if (DKV) {
                    Vec<bf16> v2;
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        v1.set2(e, a1[8 * k + e], a1[8 * k + e + 1]);
                        v2.set2(e, a2[8 * k + e] * 0.125f, a2[8 * k + e + 1] * 0.125f);
                    }
                    *reinterpret_cast<uint4*>(stg + off) = v1.v;                   // dV
                    *reinterpret_cast<uint4*>(stg + AT_TILE_BYTES + off) = v2.v;   // dK / 8
                } else {
#pragma unroll
                    for (int e = 0; e < 8; e += 2) v1.set2(e, a1[8 * k + e] * 0.125f, a1[8 * k + e + 1] * 0.125f);
                    *reinterpret_cast<uint4*>(stg + off) = v1.v;                   // dQ / 8
                }
            }
            fence_async_smem();
            named_bar(1, 256);
            if (threadIdx.x == 64) {
                if (DKV) {
                    tma_store_3d(&tmDQKV, stg, 2 * C + h * AT_HS, t * AT_BM, b);
                    tma_store_3d(&tmDQKV, stg + AT_TILE_BYTES, C + h * AT_HS, t * AT_BM, b);
                } else {
                    tma_store_3d(&tmDQKV, stg, h * AT_HS, t * AT_BM, b);
                }
                bulk_commit();
            }
            stg_pending = (gc - 1) & 1;   // read before that buffer is next written
        }
        if (threadIdx.x == 64) bulk_wait<0>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    __syncwarp();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512) : "memory");
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;
static int g_sms = 0;
static int g_at_ok = -1;
static std::mutex g_at_mutex;

int attention_tc_available() {
    std::lock_guard<std::mutex> lock(g_at_mutex);
    if (g_at_ok >= 0) return g_at_ok;
    g_at_ok = 0;
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return 0;
    if (prop.major != 10) return 0;
    g_sms = prop.multiProcessorCount;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return 0;
    g_enc = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    if (cudaFuncSetAttribute(attention_tc_forward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             AtSmem::TOTAL) != cudaSuccess)
        return 0;
    g_at_ok = 1;
    return 1;
}

// 3-D bf16 map over (cols, T, B) with row pitch `ld` elements; box {64, 128, 1}.
static bool make_map3(CUtensorMap* map, const void* base, int cols, int Tn, int B, int ld) {
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)Tn, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)ld * 2 * Tn};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int attention_tc_forward(cudaStream_t s, __nv_bfloat16* out, float* lse, const __nv_bfloat16* qkv, int B, int Tn,
                         int C, int NH, unsigned* err) {
    if (!attention_tc_available()) return GPT2_EUNSUPPORTED;
    if (C / NH != AT_HS || (((uintptr_t)qkv | (uintptr_t)out) & 15)) return GPT2_EUNSUPPORTED;
    CUtensorMap tq, to;
    if (!make_map3(&tq, qkv, 3 * C, Tn, B, 3 * C) || !make_map3(&to, out, C, Tn, B, C)) return GPT2_EUNSUPPORTED;
    const int items = ((Tn + AT_BM - 1) / AT_BM) * B * NH;
    const int grid = items < g_sms ? items : g_sms;
    attention_tc_forward_kernel<<<grid, AT_THREADS, AtSmem::TOTAL, s>>>(tq, to, lse, B, Tn, C, NH, err);
    rt_note_launches(1);
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ECUDA;
}

// 2-D fp32 map over (T, rows) with row pitch Tp (a multiple of 4, so the pitch is a
// multiple of 16 bytes); columns >= T read as zero.  Box {128, 1}; no swizzle.
static bool make_map_vec(CUtensorMap* map, const float* base, int Tn, int Tp, int rows) {
    cuuint64_t dims[2] = {(cuuint64_t)Tn, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)Tp * 4};
    cuuint32_t box[2] = {128, 1};
    cuuint32_t estr[2] = {1, 1};
    return g_enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// D[b,h,t] = sum_d dO[b,t,h,d] O[b,t,h,d] (head size 64), the row sums of the softmax
// backward, written at row pitch Tp.  Eight lanes per (b, h, t) row, one 16-byte packet
// of dO and of O each, added across the eight lanes by shuffles; rows in D's own order,
// so a warp's four results are consecutive floats (B*NH*T < 2^31: 32-bit indices).
// lse_pad (nullable): also copy the forward's LSE row (pitch T) to pitch Tp, for the
// tensor maps of the backward when T is not a multiple of 4.
__global__ void attention_rowdot_kernel(float* __restrict__ D, float* __restrict__ lse_pad,
                                        const float* __restrict__ lse, const bf16* __restrict__ dout,
                                        const bf16* __restrict__ out, int B, int Tn, int Tp, int C, int NH) {
    const int row = (int)(((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 3);
    const int sub = threadIdx.x & 7;
    const bool valid = row < B * NH * Tn;
    float s = 0.f;
    int t = 0, bh = 0;
    if (valid) {
        t = row % Tn;
        bh = row / Tn;
        const int b = bh / NH, h = bh % NH;
        const size_t o = ((size_t)b * Tn + t) * C + h * AT_HS + sub * 8;
        Vec<bf16> a = load_vec(dout + o), c = load_vec(out + o);
#pragma unroll
        for (int e = 0; e < 8; e++) s += a.get(e) * c.get(e);
    }
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    if (valid && sub == 0) {
        D[(size_t)bh * Tp + t] = s;
        if (lse_pad) lse_pad[(size_t)bh * Tp + t] = lse[row];
    }
}

template <bool DKV>
static int launch_bwd(cudaStream_t s, const CUtensorMap& tq, const CUtensorMap& tdo, const CUtensorMap& tl,
                      const CUtensorMap& td, const CUtensorMap& tdq, const float* lse, const float* D, int B, int Tn,
                      int Tp, int C, int NH, unsigned* err) {
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(attention_tc_backward_kernel<DKV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 AbSmem<DKV>::TOTAL) != cudaSuccess)
            return GPT2_ECUDA;
        attr = true;
    }
    const int items = ((Tn + AT_BM - 1) / AT_BM) * B * NH;
    const int grid = items < g_sms ? items : g_sms;
    attention_tc_backward_kernel<DKV><<<grid, AT_THREADS, AbSmem<DKV>::TOTAL, s>>>(tq, tdo, tl, td, tdq, lse, D, B,
                                                                                    Tn, Tp, C, NH, err);
    rt_note_launches(1);
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ECUDA;
}

size_t attention_tc_backward_scratch_floats(int B, int Tn, int NH) {
    const size_t Tp = (size_t)(Tn + 3) / 4 * 4;
    return 2 * (size_t)B * NH * Tp;
}

int attention_tc_backward(cudaStream_t s, __nv_bfloat16* dqkv, const __nv_bfloat16* dout, const __nv_bfloat16* qkv,
                          const __nv_bfloat16* out, const float* lse, float* scratch, int B, int Tn, int C, int NH,
                          unsigned* err) {
    if (!attention_tc_available()) return GPT2_EUNSUPPORTED;
    if (C / NH != AT_HS || C % NH ||
        (((uintptr_t)qkv | (uintptr_t)dout | (uintptr_t)dqkv | (uintptr_t)out | (uintptr_t)scratch) & 15))
        return GPT2_EUNSUPPORTED;
    // D (and, when T is not a multiple of 4, a copy of the LSE) at a row pitch of Tp
    const int Tp = (Tn + 3) / 4 * 4;
    float* D = scratch;
    float* lse_pad = (Tp != Tn) ? scratch + (size_t)B * NH * Tp : nullptr;
    const float* lse_k = lse_pad ? lse_pad : lse;
    if (!lse_pad && ((uintptr_t)lse & 15)) return GPT2_EUNSUPPORTED;
    const long long rows = (long long)B * NH * Tn;
    attention_rowdot_kernel<<<(unsigned)((rows * 8 + 255) / 256), 256, 0, s>>>(D, lse_pad, lse, dout, out, B, Tn, Tp,
                                                                              C, NH);
    rt_note_launches(1);
    if (cudaGetLastError() != cudaSuccess) return GPT2_ECUDA;
    CUtensorMap tq, tdo, tl, td, tdq;
    if (!make_map3(&tq, qkv, 3 * C, Tn, B, 3 * C) || !make_map3(&tdo, dout, C, Tn, B, C) ||
        !make_map_vec(&tl, lse_k, Tn, Tp, B * NH) || !make_map_vec(&td, D, Tn, Tp, B * NH) ||
        !make_map3(&tdq, dqkv, 3 * C, Tn, B, 3 * C))
        return GPT2_EUNSUPPORTED;
    int rc = launch_bwd<true>(s, tq, tdo, tl, td, tdq, lse_k, D, B, Tn, Tp, C, NH, err);
    if (rc != GPT2_OK) return rc;
    return launch_bwd<false>(s, tq, tdo, tl, td, tdq, lse_k, D, B, Tn, Tp, C, NH, err);
}

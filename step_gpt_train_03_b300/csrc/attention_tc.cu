// Causal flash attention for head size 64 on the sm_103a tensor cores (tcgen05, TMEM,
// TMA).
//
// ujoy.net llm.c article, section "用C语言实现LLM": causal self-attention forward and
// backward.  Per head: S = Q K^T / sqrt(64) over keys j <= t, P = softmax(S), O = P V;
// the forward keeps O and each row's log-sum-exp only.
//
// Forward kernel, persistent, one CTA per SM, 352 threads.  A work item is a pair of
// 128-query tiles of one (batch, head): tile 2p+1 (slot A) and tile 2p (slot B), which
// read the same key / value tiles 0..2p+1 (slot B stops one tile earlier), so each K
// and V tile is loaded once for both.  Items go heaviest first, dealt to the CTAs in
// snake order (forward in even rounds, backward in odd ones) to even out the tiles per
// CTA.
//   warp 0     TMA producer: the item's Q tiles (double-buffered across items), then
//              K_j and V_j through a ring of AT_RING slots
//   warp 1     TMEM owner and slot A's MMA issuer, warp 10 slot B's: S_X = Q_X K_j^T
//              (M=128, N=128, K=64) into the slot's S buffer; O_X += P_X V_j (M=128,
//              N=64, K=128) with P_X, the A operand, read from TMEM (no shared-memory
//              traffic for it); one issuing thread per slot, so neither slot's products
//              wait behind the other's in a single thread's instruction stream
//   warps 2-5  softmax of slot A, warps 6-9 softmax of slot B: one query row per
//              thread (the warp's TMEM lane quadrant), all 128 keys of a tile; the row
//              max is a thread's own, so no exchange between warps
// The two softmax warpgroups work on different tiles and are not synchronised with each
// other, so while one waits for its scores or finishes a tile, the other keeps the
// exponential unit busy, and the tensor pipe always has the other slot's products.
// The exponent reference of a row (its max so far) is only raised when a new score
// exceeds it by more than 2^8: then, and only then, the row of O in TMEM is rescaled
// (after the P V in flight has landed).  Numerator and denominator always use the same
// reference, so O / l is exact; p <= 256 stays far inside fp32 and bf16 range.
// TMEM (512 columns): S_A, S_B (128 each), O_A, O_B (64 each), P_A, P_B (bf16 pairs, 64
// each).  Every wait is bounded.  The tensor maps are 3-D (columns, T, B) so no tile
// ever reads or writes past its own sequence.
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
#define AT_RING 6                  // K / V tile slots of the forward
#define AT_TILE_BYTES (128 * 64 * 2)
#define AT_THREADS 320             // backward: loads, MMA issuer, 8 compute warps
#define AT_FWD_WARPS 11            // forward: producer, MMA issuer A, 8 softmax warps, MMA issuer B
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
    static constexpr int Q_OFF = 0;                                          // [item parity][slot]
    static constexpr int RING_OFF = Q_OFF + 4 * AT_TILE_BYTES;
    static constexpr int O_OFF = RING_OFF + AT_RING * AT_TILE_BYTES;         // [slot] output staging
    static constexpr int BAR_OFF = O_OFF + 2 * AT_TILE_BYTES;
    // q_full[2], q_empty[2], ring_full[R], ring_empty[R]; per slot s_full, s_free,
    // p_full, o_done, o_free; done; then tmem address and abort flag
    static constexpr int NBAR = 4 + 2 * AT_RING + 10 + 1;
    static constexpr int TOTAL = BAR_OFF + NBAR * 8 + 16 + 1024;
    static_assert(TOTAL <= 232448, "shared memory of one CTA");
};

__global__ void __launch_bounds__(AT_FWD_WARPS * 32, 1)
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
    uint64_t* s_full = ring_empty + AT_RING;   // [slot]
    uint64_t* s_free = s_full + 2;
    uint64_t* p_full = s_free + 2;
    uint64_t* o_done = p_full + 2;
    uint64_t* o_free = o_done + 2;
    uint64_t* done = o_free + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = B * NH;
    const int nqt = (Tn + AT_BM - 1) / AT_BM;
    const int npairs = (nqt + 1) / 2;
    const int n_items = npairs * BH;
    const int G = gridDim.x, cta = blockIdx.x;
    // the k-th item of this CTA (snake order), or -1
    auto item_at = [&](int k) -> int {
        const int it = k * G + ((k & 1) ? (G - 1 - cta) : cta);
        return it < n_items ? it : -1;
    };
    // item -> (pair p, b*h); tiles per slot: A = tile 2p+1 (when it exists), B = tile 2p
    auto decode = [&](int it, int& p, int& bh, int& nkA, int& nkB) {
        p = npairs - 1 - it / BH;
        bh = it % BH;
        nkA = (2 * p + 1 < nqt) ? 2 * p + 2 : 0;
        nkB = 2 * p + 1;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) { mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 2); }
        for (int i = 0; i < AT_RING; i++) { mbar_init(&ring_full[i], 1); mbar_init(&ring_empty[i], 2); }
        for (int x = 0; x < 2; x++) {
            mbar_init(&s_full[x], 1);
            mbar_init(&s_free[x], 4);
            mbar_init(&p_full[x], 4);
            mbar_init(&o_done[x], 1);
            mbar_init(&o_free[x], 4);
        }
        mbar_init(done, 2);
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
    // set-up done (barriers, TMEM, descriptor prefetch): wait for the predecessor's
    // results, and let the next kernel's CTAs launch onto SMs as ours retire
    pdl_wait();
    pdl_trigger();
    const uint32_t tmem_base = *tmem_slot;
    auto TM_S = [&](int x) { return tmem_base + x * AT_BN; };          // columns 0, 128
    auto TM_O = [&](int x) { return tmem_base + 256 + x * AT_HS; };    // 256, 320
    auto TM_P = [&](int x) { return tmem_base + 384 + x * 64; };       // 384, 448

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int rc = 0;
            bool ok = true;
            for (int k = 0; ok; k++) {
                const int it = item_at(k);
                if (it < 0) break;
                int p, bh, nkA, nkB;
                decode(it, p, bh, nkA, nkB);
                const int b = bh / NH, h = bh % NH;
                const int qb = k & 1;
                if (!mbar_wait(&q_empty[qb], ((k >> 1) & 1) ^ 1, abort_flag, err)) break;
                mbar_expect_tx(&q_full[qb], (nkA ? 2 : 1) * AT_TILE_BYTES);
                if (nkA)
                    tma_load_3d(smem + S::Q_OFF + (qb * 2 + 0) * AT_TILE_BYTES, &tmQKV, &q_full[qb], h * AT_HS,
                                (2 * p + 1) * AT_BM, b);
                tma_load_3d(smem + S::Q_OFF + (qb * 2 + 1) * AT_TILE_BYTES, &tmQKV, &q_full[qb], h * AT_HS,
                            2 * p * AT_BM, b);
                const int nk = nkA ? nkA : nkB;
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
    } else if (warp == 1 || warp == AT_FWD_WARPS - 1) {
        // ------------------------------------------------------------ MMA issuers
        // warp 1 issues slot A's products, the last warp slot B's: S_x = Q_x K_j^T, then
        // O_x += P_x V_{j-1}.  Both walk every K / V stage of the item (slot B has one key
        // tile fewer) and commit the shared ring, Q and done barriers once each (those
        // count two arrivals), so a stage is released when both slots' products are done.
        if (lane == 0) {
            const int x = warp == 1 ? 0 : 1;
            constexpr uint32_t IDESC_S = idesc_bf16(AT_BM, AT_BN, false, false);
            constexpr uint32_t IDESC_O = idesc_bf16(AT_BM, AT_HS, false, true);
            int rc = 0, sn = 0, pn = 0, nitems = 0;      // this slot's S, P V, items so far
            bool ok = true;
            for (int k = 0; ok; k++) {
                const int it = item_at(k);
                if (it < 0) break;
                int p, bh, nkx[2];
                decode(it, p, bh, nkx[0], nkx[1]);
                const int nk = nkx[0] ? nkx[0] : nkx[1];
                const int nkm = nkx[x];                      // this slot's key tiles (0: none)
                const int qb = k & 1;
                if (!mbar_wait(&q_full[qb], (k >> 1) & 1, abort_flag, err)) break;
                // K_j at ring index rc + 2j, V_j at rc + 2j + 1.  Order per j: S_x(j), then
                // O_x += P_x(j-1) V_{j-1}
                for (int j = 0; j <= nk && ok; j++) {
                    if (j < nk) {
                        const int kidx = rc + 2 * j, ks = kidx % AT_RING;
                        if (!mbar_wait(&ring_full[ks], (kidx / AT_RING) & 1, abort_flag, err)) { ok = false; break; }
                        if (j < nkm) {
                            if (!mbar_wait(&s_free[x], (sn & 1) ^ 1, abort_flag, err)) { ok = false; break; }
                            tc_fence_after();
                            const uint32_t k_addr = smem_u32(smem + S::RING_OFF + ks * AT_TILE_BYTES);
                            const uint32_t q_addr = smem_u32(smem + S::Q_OFF + (qb * 2 + x) * AT_TILE_BYTES);
                            // descriptors of step kk: the start address field (bytes / 16) advances by 2
                            const uint64_t qd = sdesc(q_addr, 16, 1024), kd = sdesc(k_addr, 16, 1024);
#pragma unroll
                            for (int kk = 0; kk < AT_HS / 16; kk++)
                                tc_mma(TM_S(x), qd + 2 * kk, kd + 2 * kk, IDESC_S, kk > 0 ? 1u : 0u);
                            tc_commit(&s_full[x]);
                            sn++;
                        }
                        tc_commit(&ring_empty[ks]);                  // K_j read by this slot's products
                        if (j == nk - 1) tc_commit(&q_empty[qb]);    // and its Q tile
                    }
                    if (j >= 1) {
                        const int jj = j - 1;
                        const int vidx = rc + 2 * jj + 1, vs = vidx % AT_RING;
                        if (!mbar_wait(&ring_full[vs], (vidx / AT_RING) & 1, abort_flag, err)) { ok = false; break; }
                        if (jj < nkm) {
                            if (!mbar_wait(&p_full[x], pn & 1, abort_flag, err)) { ok = false; break; }
                            // the first P V of an item overwrites O: its last readout must be done
                            if (jj == 0 && nitems > 0 &&
                                !mbar_wait(&o_free[x], (nitems - 1) & 1, abort_flag, err)) { ok = false; break; }
                            tc_fence_after();
                            const uint32_t v_addr = smem_u32(smem + S::RING_OFF + vs * AT_TILE_BYTES);
                            const uint64_t vd = sdesc(v_addr, 8192, 1024);    // step kk: + 2048 bytes
#pragma unroll
                            for (int kk = 0; kk < AT_BN / 16; kk++)
                                tc_mma_ts(TM_O(x), TM_P(x) + kk * 8, vd + 128 * kk, IDESC_O,
                                          (jj > 0 || kk > 0) ? 1u : 0u);
                            tc_commit(&o_done[x]);
                            pn++;
                        }
                        tc_commit(&ring_empty[vs]);
                    }
                }
                if (nkm) nitems++;
                rc += 2 * nk;
            }
            tc_commit(done);
            const long long t0 = clock64();
            while (!mbar_try_wait(done, 0))
                if (clock64() - t0 > TC_WAIT_LIMIT) { raise_error(err, ERRBIT_TIMEOUT); break; }
        }
    } else {
        // ------------------------------------------------------------ softmax warps 2..9
        const int x = (warp - 2) >> 2;                       // slot: 0 = A (warps 2-5), 1 = B
        const int lane_grp = warp & 3;                       // TMEM lanes 32*lane_grp .. +31
        const int r = lane_grp * 32 + lane;                  // query row in the tile
        const uint32_t lrow = (uint32_t)(lane_grp * 32) << 16;
        const int leader = 64 + 128 * x;                     // the warpgroup's store thread
        const int wg_bar = 1 + x;                            // its named barrier (128 threads)
        uint8_t* obuf = smem + S::O_OFF + x * AT_TILE_BYTES;
        const float sl2 = AT_LOG2E * 0.125f;                 // log2(e) / sqrt(64)
        int sn = 0, pn = 0, pv_seen = 0;
        bool staged = false, alive = true;
        auto wait_bar = [&](uint64_t* bar, uint32_t parity) -> bool {
            int okw = 1;
            if (lane == 0) okw = mbar_wait(bar, parity, abort_flag, err) ? 1 : 0;
            okw = __shfl_sync(0xffffffffu, okw, 0);
            __syncwarp();
            return okw != 0;
        };
        // wait until P V number n of this slot has completed (completions observed in order)
        auto wait_pv = [&](int n) -> bool {
            if (n < pv_seen) return true;
            pv_seen = n + 1;
            return wait_bar(&o_done[x], n & 1);
        };
        for (int k = 0; alive; k++) {
            const int it = item_at(k);
            if (it < 0) break;
            int p, bh, nkA, nkB;
            decode(it, p, bh, nkA, nkB);
            const int nkx = x == 0 ? nkA : nkB;
            if (nkx == 0) continue;                          // slot A of a last, odd tile
            const int b = bh / NH, h = bh % NH;
            const int qt = x == 0 ? 2 * p + 1 : 2 * p;
            const int q = qt * AT_BM + r;
            float m = -INFINITY, l = 0.f;                    // exponent reference, running sum
            for (int j = 0; j < nkx; j++) {
                // The row's 128 scores come in two halves of 64 (registers hold one half and
                // its temporaries): the first half is read for its max only, the second is
                // read and kept; after the second half's exponentials the first half is read
                // again, and the S buffer is then free for S(j+1).
                const bool diag = j == nkx - 1;              // keys after the query are masked
                auto load_half = [&](int hf, uint32_t (&v)[2][32]) {
                    tmem_ld32(TM_S(x) + lrow + hf * 64, v[0]);
                    tmem_ld32(TM_S(x) + lrow + hf * 64 + 32, v[1]);
                    tmem_ld_wait();
                    if (diag) {
#pragma unroll
                        for (int i = 0; i < 64; i++)
                            if (hf * 64 + i > r) v[i >> 5][i & 31] = __float_as_uint(-INFINITY);
                    }
                };
                auto half_max = [&](const uint32_t (&v)[2][32]) -> float {
                    float a0 = __uint_as_float(v[0][0]), a1 = __uint_as_float(v[0][1]);
                    float a2 = __uint_as_float(v[1][0]), a3 = __uint_as_float(v[1][1]);
#pragma unroll
                    for (int i = 2; i < 32; i += 2) {
                        a0 = fmax3(a0, __uint_as_float(v[0][i]), __uint_as_float(v[0][i + 1]));
                        a2 = fmax3(a2, __uint_as_float(v[1][i]), __uint_as_float(v[1][i + 1]));
                    }
                    return fmax3(a0, a2, fmaxf(a1, a3));
                };
                float rs = 0.f;
                // p = 2^(s sl2 - m) for one half: bf16 pairs into P (TMEM), partial row sum
                auto exp_half = [&](int hf, const uint32_t (&v)[2][32], float mref) {
#pragma unroll
                    for (int c8 = 0; c8 < 4; c8++) {
                        float pv[16];
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            const int e = c8 * 16 + i;
                            const float2 a = __ffma2_rn(make_float2(__uint_as_float(v[e >> 5][e & 31]),
                                                                    __uint_as_float(v[e >> 5][(e & 31) + 1])),
                                                        make_float2(sl2, sl2), make_float2(-mref, -mref));
                            pv[i] = ex2_fast(a.x);
                            pv[i + 1] = ex2_fast(a.y);
                        }
                        uint32_t pk[8];
#pragma unroll
                        for (int i = 0; i < 8; i++) {
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(pv[2 * i], pv[2 * i + 1]);
                            pk[i] = *reinterpret_cast<uint32_t*>(&h2);
                        }
                        tmem_st8(TM_P(x) + lrow + hf * 32 + c8 * 8, pk);
                        // pairwise tree sum; the levels with w >= 2 in packed pairs
#pragma unroll
                        for (int w = 8; w > 1; w >>= 1)
#pragma unroll
                            for (int i = 0; i < w; i += 2) {
                                const float2 s2 = __fadd2_rn(make_float2(pv[i], pv[i + 1]),
                                                             make_float2(pv[i + w], pv[i + w + 1]));
                                pv[i] = s2.x;
                                pv[i + 1] = s2.y;
                            }
                        rs += pv[0] + pv[1];
                    }
                };
                if (!wait_bar(&s_full[x], sn & 1)) { alive = false; break; }
                tc_fence_after();
                float mx;
                uint32_t sv[2][32];
                load_half(0, sv);
                mx = half_max(sv);
                load_half(1, sv);
                mx = fmaxf(mx, half_max(sv)) * sl2;          // scaling by sl2 > 0 keeps the max
                const bool raise = mx > m + AT_RESCALE_LOG2;
                const float m_new = raise ? mx : m;
                const float corr = ex2_fast(m - m_new);      // 1 when unchanged, 0 on the first tile
                if (__any_sync(0xffffffffu, raise && j > 0)) {
                    // rescale this warp's rows of O once the P V in flight has landed
                    if (!wait_pv(pn - 1)) { alive = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int hh = 0; hh < 2; hh++) {
                        uint32_t rr[32];
                        tmem_ld32(TM_O(x) + lrow + hh * 32, rr);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; i++) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * corr);
                        tmem_st32(TM_O(x) + lrow + hh * 32, rr);
                    }
                    tmem_st_wait();
                }
                m = m_new;
                // P of this tile goes where the previous tile's P was read by P V
                if (j > 0 && !wait_pv(pn - 1)) { alive = false; break; }
                tc_fence_after();
                exp_half(1, sv, m);
                load_half(0, sv);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[x]);
                sn++;
                exp_half(0, sv, m);
                l = l * corr + rs;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[x]);
                pn++;
            }
            // the item's last P V, then normalise and write this row of O
            // (after an abort the reads below see whatever TMEM holds and nothing is stored)
            const bool okw = alive && wait_pv(pn - 1);
            tc_fence_after();
            float o[64];
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                uint32_t rr[32];
                tmem_ld32(TM_O(x) + lrow + hh * 32, rr);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; i++) o[hh * 32 + i] = __uint_as_float(rr[i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && okw) mbar_arrive(&o_free[x]);
            const float inv = 1.0f / l;
            // the previous item's store must have finished reading the staging buffer; the
            // warpgroup leaves together if any of its warps gave up waiting
            if (staged && threadIdx.x == leader) bulk_wait_read<0>();
            if (!named_bar_and(wg_bar, 128, okw)) break;
#pragma unroll
            for (int ch = 0; ch < 8; ch++) {
                Vec<bf16> ov;
#pragma unroll
                for (int e = 0; e < 8; e += 2) ov.set2(e, o[8 * ch + e] * inv, o[8 * ch + e + 1] * inv);
                *reinterpret_cast<uint4*>(obuf + r * 128 + ((ch ^ (r & 7)) << 4)) = ov.v;
            }
            fence_async_smem();
            named_bar(wg_bar, 128);
            if (threadIdx.x == leader) {
                tma_store_3d(&tmO, obuf, h * AT_HS, qt * AT_BM, b);
                bulk_commit();
            }
            staged = true;
            if (q < Tn) lse[(size_t)bh * Tn + q] = (m + log2f(l)) / AT_LOG2E;
        }
        if (threadIdx.x == leader) bulk_wait<0>();
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
// Warp 0 loads (the item's two row tiles once; the per-u tiles through a ring with, in
// DKV mode, that u's LSE and D vectors); warp 1 issues the MMAs (the next S/dP pair is
// issued before the dV/dK (dQ) products of the current one); warps 2-9 compute, two warps
// per TMEM lane quadrant, each on half the columns of a tile (a TMEM lane is a key row in
// DKV mode, a query row in DQ mode).  The operands the compute warps produce for the
// N = 64 products -- P^T and dS^T (DKV), dS (DQ), bf16 pairs -- go to TMEM and are read
// there as the A operand, so those products fetch only their 64-wide B operand from
// shared memory.  TMEM (512 columns): S (S^T) 128, dP (dP^T) 128, dV or dQ 64, dK 64, then
// DKV: P^T 64 and dS^T 64 (single-buffered: the compute warps compute half a tile before
// they need the buffer back); DQ: dS 2 x 64 (double-buffered).
#define AB_STAGE_BYTES (2 * AT_TILE_BYTES + 1024)   // two tiles + LSE[128] + D[128]

template <bool DKV>
struct AbSmem {
    static constexpr int RING = 4;
    static constexpr int R_OFF = 0;                                        // 2 row tiles
    static constexpr int RING_OFF = R_OFF + 2 * AT_TILE_BYTES;
    static constexpr int STG_OFF = RING_OFF + RING * AB_STAGE_BYTES;       // output staging, 2 tiles
    static constexpr int BAR_OFF = STG_OFF + 2 * AT_TILE_BYTES;
    // rr_full, rr_empty, ring_full[RING], ring_empty[RING], x_full, x_free, pds_full[2],
    // pds_free[2], acc_free, done; tmem address, abort flag
    static constexpr int NBAR = 2 + 2 * RING + 8;
    static constexpr int TOTAL = BAR_OFF + NBAR * 8 + 16 + 1024;
    static_assert(TOTAL <= 232448, "shared memory of one CTA");
    static constexpr int NPB = DKV ? 1 : 2;          // P / dS buffers in TMEM
};

template <bool DKV>
__global__ void __launch_bounds__(AT_THREADS, 1)
attention_tc_backward_kernel(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmDO,
                             const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmD,
                             const __grid_constant__ CUtensorMap tmDQKV, const float* __restrict__ lse,
                             const float* __restrict__ Dsum, float* __restrict__ bsum, int B, int Tn, int Tp, int C,
                             int NH, unsigned* err) {
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
    // set-up done (barriers, TMEM, descriptor prefetch): wait for the predecessor's
    // results, and let the next kernel's CTAs launch onto SMs as ours retire
    pdl_wait();
    pdl_trigger();
    const uint32_t tmem_base = *tmem_slot;
    // S (S^T), dP (dP^T), dV or dQ, dK; then DKV: P^T, dS^T; DQ: dS[2]
    const uint32_t TM_X1 = tmem_base, TM_X2 = tmem_base + 128, TM_A1 = tmem_base + 256, TM_A2 = tmem_base + 320;
    const uint32_t TM_P = tmem_base + 384;
    auto TM_DS = [&](int pb) { return tmem_base + (DKV ? 448 : 384 + 64 * pb); };

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
            int rc = 0, xc = 0, gc = 0, local = 0;
            bool ok = true;
            // the S / dP pair for the ring stage of index `idx`
            auto issue_x = [&](int idx) -> bool {
                const int slot = idx % AB_RING;
                if (!mbar_wait(&ring_full[slot], (idx / AB_RING) & 1, abort_flag, err)) return false;
                if (!mbar_wait(x_free, (xc & 1) ^ 1, abort_flag, err)) return false;
                tc_fence_after();
                const uint32_t st = smem_u32(smem + S::RING_OFF + slot * AB_STAGE_BYTES);
                // descriptors of step k: the start address field (bytes / 16) advances by 2
                const uint64_t d0 = sdesc(r0, 16, 1024), d1 = sdesc(r1, 16, 1024);
                const uint64_t e0 = sdesc(st, 16, 1024), e1 = sdesc(st + AT_TILE_BYTES, 16, 1024);
#pragma unroll
                for (int k = 0; k < AT_HS / 16; k++) tc_mma(TM_X1, d0 + 2 * k, e0 + 2 * k, IDESC_X, k > 0);
#pragma unroll
                for (int k = 0; k < AT_HS / 16; k++) tc_mma(TM_X2, d1 + 2 * k, e1 + 2 * k, IDESC_X, k > 0);
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
                    const int pb = gc % S::NPB;                      // P / dS buffer of this tile
                    if (!mbar_wait(&pds_full[pb], (gc / S::NPB) & 1, abort_flag, err)) { ok = false; break; }
                    if (i == 0 && local > 0 && !mbar_wait(acc_free, (local - 1) & 1, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    if (DKV) {
                        // dV += P^T dO_u ; dK += dS^T Q_u (A operands from TMEM, 8 columns per 16 queries)
                        const uint64_t bo = sdesc(st + AT_TILE_BYTES, 8192, 1024), bq = sdesc(st, 8192, 1024);
#pragma unroll
                        for (int k = 0; k < AT_BN / 16; k++) {      // step k: + 2048 bytes
                            tc_mma_ts(TM_A1, TM_P + k * 8, bo + 128 * k, IDESC_A, (i > 0 || k > 0));
                            tc_mma_ts(TM_A2, TM_DS(pb) + k * 8, bq + 128 * k, IDESC_A, (i > 0 || k > 0));
                        }
                    } else {
                        // dQ += dS K_u (dS from TMEM)
                        const uint64_t bk = sdesc(st, 8192, 1024);
#pragma unroll
                        for (int k = 0; k < AT_BN / 16; k++)
                            tc_mma_ts(TM_A1, TM_DS(pb) + k * 8, bk + 128 * k, IDESC_A, (i > 0 || k > 0));
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
        uint8_t* stg = smem + S::STG_OFF;
        int rc = 0, xc = 0, gc = 0, local = 0;
        int pf_seen[2] = {0, 0};                            // pds_free completions observed per buffer
        bool stg_pending = false;                           // an item's output store may still read stg
        bool alive = true;
        auto wait_one = [&](uint64_t* bar, uint32_t parity) -> bool {
            int okw = 1;
            if (lane == 0) okw = mbar_wait(bar, parity, abort_flag, err) ? 1 : 0;
            okw = __shfl_sync(0xffffffffu, okw, 0);
            __syncwarp();
            return okw != 0;
        };
        // wait for the dV/dK (dQ) products of tile n: completion n / NPB of buffer n % NPB's
        // barrier (each buffer's completions are observed in order)
        auto wait_pds_free = [&](int n) -> bool {
            const int b = n % S::NPB, need = n / S::NPB + 1;
            if (pf_seen[b] >= need) return true;
            pf_seen[b] = need;
            return wait_one(&pds_free[b], (n / S::NPB) & 1);
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
                const int pb = gc % S::NPB;
#pragma unroll 1
                for (int ci = 0; ci < 2; ci++) {
                    const int c = half * 64 + ci * 32;      // first column of this chunk
                    uint32_t s1[32], s2[32];
                    tmem_ld32(TM_X1 + lrow + c, s1);
                    tmem_ld32(TM_X2 + lrow + c, s2);
                    tmem_ld_wait();
                    if (ci == 1) {
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
                    // the products of tile gc - NPB must have read this tile's buffers (checked
                    // once, after the first chunk's arithmetic)
                    if (ci == 0 && gc >= S::NPB) {
                        if (!wait_pds_free(gc - S::NPB)) { alive = false; break; }
                        tc_fence_after();
                    }
                    // bf16 pairs along the row: 16 TMEM columns per 32 values
                    uint32_t pk[16];
#pragma unroll
                    for (int k = 0; k < 16; k++) {
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(ds[2 * k], ds[2 * k + 1]);
                        pk[k] = *reinterpret_cast<uint32_t*>(&h2);
                    }
                    tmem_st16(TM_DS(pb) + lrow + (c >> 1), pk);
                    if (DKV) {
#pragma unroll
                        for (int k = 0; k < 16; k++) {
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(p[2 * k], p[2 * k + 1]);
                            pk[k] = *reinterpret_cast<uint32_t*>(&h2);
                        }
                        tmem_st16(TM_P + lrow + (c >> 1), pk);
                    }
                }
                if (!alive) break;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&pds_full[pb]);
            }
            // accumulators of the item: wait for its last products, read, release, store
            // (after an abort the reads below see whatever TMEM holds and nothing is stored)
            const bool okw = alive && wait_pds_free(gc - 1);
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
            if (lane == 0 && okw) mbar_arrive(acc_free);
            // the previous item's store must have finished reading the staging buffers; the
            // compute warps leave together if any of them gave up waiting
            if (stg_pending && threadIdx.x == 64) bulk_wait_read<0>();
            if (!named_bar_and(1, 256, okw)) break;
            // stage 128B-swizzled rows, then TMA-store
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
            stg_pending = true;
            if (bsum) {
                // the qkv bias gradient: column sums of the staged (stored) tiles over 32
                // rows, one partial row per (batch, row tile, row quarter).  Thread: a
                // column pair of the dV or dK tile (dQ: warps 0-3 only) and a row quarter
                const int ct = threadIdx.x - 64;                     // 0..255
                const int tile = ct >> 7, quarter = (ct >> 5) & 3, cp = lane;
                if (DKV || tile == 0) {
                    const uint8_t* tb = stg + tile * AT_TILE_BYTES;
                    // rows past T are left out (their staged values are not defined)
                    const int nrow = Tn - t * AT_BM - quarter * 32;
                    float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int hb = 0; hb < 2; hb++) {
                        float2 p[16];
#pragma unroll
                        for (int k = 0; k < 16; k++) {
                            const int i = hb * 16 + k, rr = quarter * 32 + i;
                            const uint32_t u = *reinterpret_cast<const uint32_t*>(
                                tb + rr * 128 + (((cp >> 2) ^ (rr & 7)) << 4) + (cp & 3) * 4);
                            p[k] = i < nrow ? make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u))
                                            : make_float2(0.f, 0.f);
                        }
#pragma unroll
                        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                            for (int k = 0; k < w; k++) p[k] = __fadd2_rn(p[k], p[k + w]);
                        acc2 = __fadd2_rn(acc2, p[0]);
                    }
                    // column offset within dqkv's row: dQ at 0, dK at C, dV at 2C
                    const int part = DKV ? (tile == 0 ? 2 : 1) : 0;
                    float* prow = bsum + ((size_t)(b * nt + t) * 4 + quarter) * 3 * C + part * C + h * AT_HS + 2 * cp;
                    *reinterpret_cast<float2*>(prow) = acc2;
                }
            }
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
    const int items = ((Tn + AT_BM - 1) / AT_BM + 1) / 2 * B * NH;      // pairs of query tiles
    const int grid = items < g_sms ? items : g_sms;
    launch_pdl(attention_tc_forward_kernel, grid, AT_FWD_WARPS * 32, AtSmem::TOTAL, s, tq, to, lse, B, Tn, C, NH, err);
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
    pdl_wait();
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
                      const CUtensorMap& td, const CUtensorMap& tdq, const float* lse, const float* D, float* bsum,
                      int B, int Tn, int Tp, int C, int NH, unsigned* err) {
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(attention_tc_backward_kernel<DKV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 AbSmem<DKV>::TOTAL) != cudaSuccess)
            return GPT2_ECUDA;
        attr = true;
    }
    const int items = ((Tn + AT_BM - 1) / AT_BM) * B * NH;
    const int grid = items < g_sms ? items : g_sms;
    launch_pdl(attention_tc_backward_kernel<DKV>, grid, AT_THREADS, AbSmem<DKV>::TOTAL, s, tq, tdo, tl, td, tdq, lse, D, bsum,
               B, Tn, Tp, C, NH, err);
    rt_note_launches(1);
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ECUDA;
}

size_t attention_tc_backward_scratch_floats(int B, int Tn, int NH) {
    const size_t Tp = (size_t)(Tn + 3) / 4 * 4;
    return 2 * (size_t)B * NH * Tp;
}

int attention_tc_backward(cudaStream_t s, __nv_bfloat16* dqkv, const __nv_bfloat16* dout, const __nv_bfloat16* qkv,
                          const __nv_bfloat16* out, const float* lse, float* scratch, float* bias_partial, int B,
                          int Tn, int C, int NH, unsigned* err) {
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
    launch_pdl(attention_rowdot_kernel, (unsigned)((rows * 8 + 255) / 256), 256, 0, s, D, lse_pad, lse, dout, out, B, Tn, Tp,
                                                                              C, NH);
    rt_note_launches(1);
    if (cudaGetLastError() != cudaSuccess) return GPT2_ECUDA;
    CUtensorMap tq, tdo, tl, td, tdq;
    if (!make_map3(&tq, qkv, 3 * C, Tn, B, 3 * C) || !make_map3(&tdo, dout, C, Tn, B, C) ||
        !make_map_vec(&tl, lse_k, Tn, Tp, B * NH) || !make_map_vec(&td, D, Tn, Tp, B * NH) ||
        !make_map3(&tdq, dqkv, 3 * C, Tn, B, 3 * C))
        return GPT2_EUNSUPPORTED;
    int rc = launch_bwd<true>(s, tq, tdo, tl, td, tdq, lse_k, D, bias_partial, B, Tn, Tp, C, NH, err);
    if (rc != GPT2_OK) return rc;
    return launch_bwd<false>(s, tq, tdo, tl, td, tdq, lse_k, D, bias_partial, B, Tn, Tp, C, NH, err);
}

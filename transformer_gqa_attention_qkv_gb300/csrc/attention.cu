// attention.cu -- causal grouped-query flash attention on tcgen05 (prefill).
//
// Computes, for query head j, KV head g = j / G (G = Hq/Hkv), query position t:
//   attn[b, t, j*d:(j+1)*d] = softmax_u( <q, k_u> / sqrt(d) ) v_u   over u <= t
// ([T07] §4 step 6 in fp32; [NeoX] "Scaling and RoPE" scale head_dim^-0.5;
//  [NeoX] "Attention output flattening": output width Hq*d).
//
// Work item: (sequence b, KV head g, block of 2R positions), R = 128/G.  The G
// query heads of the group are packed into the MMA's M dimension: row r of a
// 128-row tile is head g*G + r/R at position t0 + r%R.  A CTA owns two such
// tiles (positions t0.., t0+R..); every K/V tile of 128 keys is brought into
// shared memory once by TMA and used by all G heads of both tiles.
//
//   warp 0      TMA: both Q tiles once, then K and V tiles into a ring
//   warp 1      MMA: per key tile j, for tile i = 0, 1:
//                 O_i += P_i(j) V(j)  (P read from TMEM),  S_i(j+1) = Q_i K(j+1)^T
//   warps 2..5  softmax of tile 0, warps 6..9 softmax of tile 1 (one thread per
//               row; tcgen05.ld 32x32b gives a thread a whole row, so the row
//               max and sum need no shuffles).  While one warpgroup runs its
//               softmax, the tensor core works on the other tile.
//
// TMEM (512 columns): tile i holds S_i in columns [256i, 256i+128) and O_i in
// [256i+128, 256i+128+d') (d' = d rounded up to 64 or 128).  P_i (binary16, two per column) is written over the
// first 64 columns of S_i and consumed from there by the PV MMA; MMAs issued by
// one thread run in order, so S_i(j+1) overwrites P_i(j) only after PV_i(j).
//
// Online softmax in fp32 with exp2 and the scale folded into log2 units.  O is
// rescaled in TMEM only when a row's running max grows by more than 2^8; P
// stays <= 2^8 in between, and the final O / l is exact either way.
//
// Cached variant with kv_splits > 1: the keys of a work item are split into
// kv_splits consecutive ranges of key tiles, each its own work item (a grid of
// few, equally long items otherwise leaves most SMs idle in its last wave);
// each writes its rows' O normalised by its own row sum (binary16) and its
// log2-sum-exp, and combine_kernel merges them.
//
// Q, K and V arrive as binary16: with QK-norm their rows are bounded by
// sqrt(d) * max|w|, and binary16 keeps 3 more mantissa bits than bf16, which
// cuts the rounding error that storage adds to scores and outputs.  The
// cached variant reads a binary16 copy of the bf16 cache rows it attends
// (made by cache_widen_kernel, exact for every bf16 value below 2^16), so Q
// and P stay binary16 there too.
#include "internal.h"
#include "ptx.cuh"

namespace gqa {

namespace {

// TMEM -> registers, 32 lanes x 32 bits, 128 consecutive columns, then wait;
// *mx is this thread's maximum over the 128 values (the load reduces them as it
// reads: tcgen05.ld.red, checked per lane against the loaded values).
__device__ __forceinline__ void tmem_ld128_max(uint32_t taddr, uint32_t (&r)[128], float &mx)
{
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x128.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, %128, [%129];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), 
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), 
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), 
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), 
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), 
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), 
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), 
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), 
          "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), 
          "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), 
          "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), 
          "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), 
          "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), 
          "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), 
          "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), 
          "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127]), 
          "=f"(mx)
        : "r"(taddr)
        : "memory");
}

// L2 residency hints for the tensor copies: K and V tiles are read again by
// every later query block of their KV head, Q and the output stream through
// once, so K/V are kept (evict_last) and Q goes first (evict_first).
__device__ __forceinline__ uint64_t l2_policy_keep()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_stream()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void tma_load_3d_hint(void *dst, const CUtensorMap *tm, int x, int y, int z, uint64_t *bar,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"((uint64_t)tm), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

constexpr int kRows = 128;      // MMA M: packed query rows per tile
constexpr int kKeys = 128;      // keys per K/V tile
constexpr int kTiles = 2;       // query tiles per CTA
constexpr int kThreads = 320;   // 2 + 2 x 4 warps
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only past a 256x growth

struct AttnParams {
    int B, S, Hq, Hkv, G, R, n_qblk, causal, num_items;
    int kv_seq;            // sequence extent of the K/V tensors
    const int *kv_start;   // device [B]: cached keys before the queries (NULL: none)
    float scale_log2;  // log2(e) / sqrt(d)
    uint16_t *out;
    float *lse;        // optional log2-sum-exp at lse[(b*Hq + head)*lse_ld + t] (plain prefill)
    int lse_ld;
    int kv_splits;        // cached variant: key ranges per query block (1: none)
    uint16_t *part_o;     // kv_splits > 1: [split][B, S, Hq*d] binary16, O / l of the split
    float *part_lse;      // kv_splits > 1: [split][B*Hq, S] log2-sum-exp of the split (-inf: no key)
    unsigned *err;
};

// Head widths that are not a multiple of 64 (80, 96) are staged as 128-wide
// rows whose columns past d are filled with zeros by the tensor copy; S
// contracts over the d real columns only, PV runs 128 wide (the zero columns
// of V give zero columns of O, which are not stored).
template <int D>
constexpr int padded_d() { return D <= 64 ? 64 : 128; }

template <int D>
struct ASmem {
    static constexpr int CHUNK = kRows * 128;             // 128 rows x 64 16-bit = 16 KB
    static constexpr int NCH = padded_d<D>() / 64;        // 64-wide d chunks
    static constexpr int STAGES = NCH == 2 ? 2 : 3;       // K/V ring depth (also keeps 1 CTA per SM)
    static constexpr int Q = 0;
    static constexpr int K = Q + kTiles * NCH * CHUNK;
    static constexpr int V = K + STAGES * NCH * CHUNK;
    static constexpr int BARS = V + STAGES * NCH * CHUNK;
    // q_full, k_full[S], v_full[S], kv_empty[S], s_full[2], p_full[2], o_done[2], drain
    static constexpr int NBARS = 1 + 3 * STAGES + 2 + 2 + 2 + 1;
    static constexpr int TMEM_SLOT = BARS + NBARS * 8;
    static constexpr int TOTAL = TMEM_SLOT + 16;
    static constexpr int ALLOC = TOTAL + 1024;
};

// D: head_dim (64, 80, 96, 128).  Q, K, V and P are binary16 in the MMAs.
// CACHED: the queries follow kv_start[b] cached keys (K and V: the binary16
// copy of a bf16 cache that cache_widen_kernel makes, kv_seq rows per head);
// otherwise the keys are exactly the S query positions (this variant compiles
// without any offset arithmetic).
template <int D, bool CACHED>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const AttnParams P)
{
    using L = ASmem<D>;
    constexpr int ST = L::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS);
    uint64_t *q_full = bars;
    uint64_t *k_full = bars + 1;
    uint64_t *v_full = k_full + ST;
    uint64_t *kv_empty = v_full + ST;
    uint64_t *s_full = kv_empty + ST;
    uint64_t *p_full = s_full + 2;
    uint64_t *o_done = p_full + 2;
    uint64_t *drain = o_done + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::TMEM_SLOT);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    unsigned *err = P.err;
    grid_dep_launch();  // the next kernel may start its prologue meanwhile

    // heavy (late) query blocks first; the key splits of one block adjacent
    const int KSPL = CACHED ? P.kv_splits : 1;
    const int split = (int)blockIdx.x % KSPL;
    const int item = (int)blockIdx.x / KSPL;
    const int bh = item % (P.B * P.Hkv);
    const int qblk = P.n_qblk - 1 - item / (P.B * P.Hkv);
    const int b = bh / P.Hkv, g = bh % P.Hkv;
    const int t0 = qblk * kTiles * P.R;
    const int t_last = min(t0 + kTiles * P.R, P.S) - 1;
    // keys [0, p0) are cached before the S queries; query t sits at position p0 + t
    int p0 = 0;
    bool bad = false;
    if constexpr (CACHED) {
        p0 = P.kv_start[b];
        bad = p0 < 0 || p0 + P.S > P.kv_seq;
        if (bad) {
            if (threadIdx.x == 0) atomicOr(P.err, kErrIndex);
            p0 = 0;
        }
    }
    const int n_all = bad ? 0 : (P.causal ? ((p0 + t_last) / kKeys + 1) : (p0 + P.S + kKeys - 1) / kKeys);
    // this item's key tiles: [kb0, kb0 + n_kv) (loop indices below are local)
    const int kb0 = split * n_all / KSPL;
    const int n_kv = (split + 1) * n_all / KSPL - kb0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::NBARS; ++i) mbar_init(bars + i, 1);
        mbar_init(p_full, 4);  // one arrival per softmax warp
        mbar_init(p_full + 1, 4);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dep_wait();  // Q, K, V come from the previous kernel (cached keys from earlier ones)

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t keep = l2_policy_keep(), stream = l2_policy_stream();
            const uint32_t q_bytes = kTiles * L::NCH * 64 * 2 * P.R * P.G;
            mbar_arrive_expect_tx(q_full, q_bytes);
            for (int i = 0; i < kTiles; ++i)
                for (int c = 0; c < L::NCH; ++c)
                    tma_load_3d_hint(smem + L::Q + (i * L::NCH + c) * L::CHUNK, &tmQ, c * 64, t0 + i * P.R,
                                     b * P.Hq + g * P.G, q_full, stream);
            int j = 0;
            for (; j < n_kv; ++j) {
                const int s = j % ST;
                if (!mbar_wait(kv_empty + s, ((j / ST) & 1) ^ 1, err)) break;
                mbar_arrive_expect_tx(k_full + s, L::NCH * L::CHUNK);
                for (int c = 0; c < L::NCH; ++c)
                    tma_load_3d_hint(smem + L::K + (s * L::NCH + c) * L::CHUNK, &tmK, c * 64, (kb0 + j) * kKeys,
                                     b * P.Hkv + g, k_full + s, keep);
                mbar_arrive_expect_tx(v_full + s, L::NCH * L::CHUNK);
                for (int c = 0; c < L::NCH; ++c)
                    tma_load_3d_hint(smem + L::V + (s * L::NCH + c) * L::CHUNK, &tmV, c * 64, (kb0 + j) * kKeys,
                                     b * P.Hkv + g, v_full + s, keep);
            }
            // every issued copy has landed before the CTA may exit
            mbar_wait(q_full, 0, err);
            for (int i = max(0, j - ST); i < j; ++i) {
                mbar_wait(k_full + i % ST, (i / ST) & 1, err);
                mbar_wait(v_full + i % ST, (i / ST) & 1, err);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // S: Q, K K-major over d; O: P from TMEM, V MN-major (d contiguous)
            constexpr uint32_t idesc_s = idesc_f16_f32(kRows, kKeys, 0, 0);
            constexpr int DP = padded_d<D>();
            constexpr uint32_t idesc_o = idesc_f16_f32(kRows, DP, 0, 1);
            auto issue_s = [&](int i, int j) {  // S_i = Q_i K(j)^T
                const uint32_t sQ = smem_u32(smem + L::Q + i * L::NCH * L::CHUNK);
                const uint32_t sK = smem_u32(smem + L::K + (j % ST) * L::NCH * L::CHUNK);
#pragma unroll
                for (int c = 0; c < L::NCH; ++c)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (c * 64 + k * 16 < D)  // d real columns, 16 per step
                            umma_f16_ss(tmem + 256 * i, sw128_desc(sQ + c * L::CHUNK + 32 * k, 16, 1024),
                                        sw128_desc(sK + c * L::CHUNK + 32 * k, 16, 1024), idesc_s, (c | k) != 0);
                umma_commit(s_full + i);
            };
            bool ok = (!CACHED || n_kv > 0) && mbar_wait(q_full, 0, err) && mbar_wait(k_full, 0, err);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                issue_s(1, 0);
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                const int s = j % ST;
                const uint32_t sV = smem_u32(smem + L::V + s * L::NCH * L::CHUNK);
                for (int i = 0; i < kTiles; ++i) {
                    if (!mbar_wait(p_full + i, j & 1, err)) {
                        ok = false;
                        break;
                    }
                    if (i == 0 && !mbar_wait(v_full + s, (j / ST) & 1, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tS = tmem + 256 * i, tO = tS + 128;
#pragma unroll
                    for (int k = 0; k < kKeys / 16; ++k)  // 16 keys = 8 packed TMEM columns of P
                        umma_f16_ts(tO, tS + 8 * k, sw128_desc(sV + k * 16 * 128, L::CHUNK, 1024), idesc_o,
                                    (j | k) != 0);
                    if (i == kTiles - 1) umma_commit(kv_empty + s);
                    if (j + 1 < n_kv) {
                        if (i == 0) {
                            if (!mbar_wait(k_full + (j + 1) % ST, ((j + 1) / ST) & 1, err)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        issue_s(i, j + 1);
                    } else {
                        umma_commit(o_done + i);
                    }
                }
            }
            umma_commit(drain);
            mbar_wait(drain, 0, err);
        }
    } else {
        const int wg = (warp - 2) >> 2;   // which query tile
        const int quarter = warp & 3;     // TMEM lanes this warp may access
        const int r = quarter * 32 + lane;
        const int hl = r / P.R, tl = r - hl * P.R;
        const bool in_pack = hl < P.G;
        const int t = t0 + wg * P.R + tl;
        const bool row_ok = in_pack && t < P.S;
        // keys u <= lim are visible to this row
        const int lim = !in_pack ? -1 : (P.causal ? p0 + min(t, P.S - 1) : p0 + P.S - 1);
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + 256 * wg + lane_off, tO = tS + 128;
        const float sl = P.scale_log2;
        float m_i = -INFINITY, l_i = 0.0f;

        for (int j = 0; j < n_kv; ++j) {
            if (!mbar_wait(s_full + wg, j & 1, err)) break;
            tc_fence_after();
            const int u0 = (kb0 + j) * kKeys;
            // the whole S row in registers with its maximum (one reducing TMEM load, one wait)
            uint32_t v[kKeys];
            float mx;
            tmem_ld128_max(tS, v, mx);
            if (u0 + kKeys - 1 > lim) {  // diagonal or ragged tile: mask keys past lim, max of the rest
#pragma unroll
                for (int e = 0; e < kKeys; ++e)
                    if (u0 + e > lim) v[e] = __float_as_uint(-INFINITY);
                // four independent chains of three-input max
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < kKeys; e += 8)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mx4[k] = fmax3(mx4[k], __uint_as_float(v[e + 2 * k]), __uint_as_float(v[e + 2 * k + 1]));
                mx = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]);
            }
            const float m_cand = fmaxf(m_i, mx * sl);
            float m_new = m_i, alpha = 1.0f;
            if (m_cand > m_i + kRescaleThreshold) {
                m_new = m_cand;
                alpha = ex2(m_i - m_new);  // 0 on the first tile
            }
            const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
            // p = 2^(s*scale - m) (masked keys give 2^-inf = 0), row sum, and P as
            // binary16 over the first 64 columns of S (already read)
            const float2 sl2 = make_float2(sl, sl), nm2 = make_float2(-m_use, -m_use);
            float2 rs2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float2 x = __ffma2_rn(
                        make_float2(__uint_as_float(v[32 * c + 2 * e]), __uint_as_float(v[32 * c + 2 * e + 1])), sl2,
                        nm2);
                    const float2 p = make_float2(ex2(x.x), ex2(x.y));
                    rs2[e & 1] = __fadd2_rn(rs2[e & 1], p);
                    pk[e] = pack_f16(p.x, p.y);
                }
                tmem_st16_nowait(tS + 16 * c, pk);
            }
            tmem_st_wait();
            const float rs = (rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y);
            l_i = l_i * alpha + rs;
            m_i = m_new;
            // O_i(j-1) is complete: S_i(j) was issued after PV_i(j-1)
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(tO + c, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(tO + c, o);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(p_full + wg);
        }
        const int head = g * P.G + hl;
        const size_t row = (size_t)(b * P.S + t) * P.Hq + head;  // output row, [B, S, Hq] order
        const bool split_out = CACHED && KSPL > 1;
        if (CACHED && n_kv == 0) {
            // no keys for this item: a rejected offset (reported; zero rows) or an
            // empty key split (weight zero in the combine); nothing else ran
            if (row_ok) {
                uint16_t *dst = split_out ? P.part_o + (size_t)split * P.B * P.S * P.Hq * D + row * D
                                          : P.out + row * D;
                uint4 *d4 = reinterpret_cast<uint4 *>(dst);
                for (int c = 0; c < D / 8; ++c) d4[c] = make_uint4(0, 0, 0, 0);
                if (split_out) P.part_lse[((size_t)split * P.B * P.Hq + b * P.Hq + head) * P.S + t] = -INFINITY;
            }
        } else if (mbar_wait(o_done + wg, 0, err)) {
            tc_fence_after();
            const float inv_l = (l_i > 0.0f) ? 1.0f / l_i : 0.0f;
            uint16_t *dst = split_out ? P.part_o + (size_t)split * P.B * P.S * P.Hq * D + row * D : P.out + row * D;
            if (!CACHED && P.lse && row_ok) P.lse[(size_t)(b * P.Hq + head) * P.lse_ld + t] = m_i + log2f(l_i);
            if (split_out && row_ok)
                P.part_lse[((size_t)split * P.B * P.Hq + b * P.Hq + head) * P.S + t] =
                    l_i > 0.0f ? m_i + log2f(l_i) : -INFINITY;
            bool clamped = false;
            constexpr int CW = D % 32 == 0 ? 32 : 16;  // columns per TMEM load, tiling d
#pragma unroll 1
            for (int c = 0; c < D; c += CW) {
                uint32_t o[CW];
                if constexpr (CW == 32)
                    tmem_ld32(tO + c, o);
                else
                    tmem_ld16(tO + c, o);
                if (row_ok) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
                    for (int i = 0; i < CW / 8; ++i) {
                        uint32_t w[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            float lo = __uint_as_float(o[8 * i + 2 * k]) * inv_l;
                            float hi = __uint_as_float(o[8 * i + 2 * k + 1]) * inv_l;
                            if (split_out) {  // binary16 partials: clamp to its range (reported)
                                if (fabsf(lo) > 65504.0f || fabsf(hi) > 65504.0f) {
                                    clamped = true;
                                    lo = fminf(fmaxf(lo, -65504.0f), 65504.0f);
                                    hi = fminf(fmaxf(hi, -65504.0f), 65504.0f);
                                }
                                w[k] = pack_f16(lo, hi);
                            } else {
                                w[k] = pack_bf16(lo, hi);
                            }
                        }
                        d4[i] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            if (clamped) atomicOr(P.err, kErrRange);
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Merges the key splits of the cached variant, one thread per 8 output
// values: out = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M), M = max_s lse_s
// (a split without keys has lse = -inf and weight 0).
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const AttnParams P, int rows)
{
    grid_dep_launch();
    grid_dep_wait();  // the split partials come from the attention kernel
    constexpr int TPR = D / 8;  // threads per (token, head) row
    const int gt = blockIdx.x * blockDim.x + threadIdx.x;
    const int r = gt / TPR, c8 = (gt - r * TPR) * 8;
    if (r >= rows) return;  // rows = B*S*Hq in [B, S, Hq] order
    const int head = r % P.Hq, bt = r / P.Hq;
    const int b = bt / P.S, t = bt - b * P.S;
    const size_t split_o = (size_t)P.B * P.S * P.Hq * D, split_l = (size_t)P.B * P.Hq * P.S;
    const size_t li = (size_t)(b * P.Hq + head) * P.S + t;
    float M = -INFINITY;
    for (int s = 0; s < P.kv_splits; ++s) M = fmaxf(M, P.part_lse[s * split_l + li]);
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0}, wsum = 0.0f;
    if (M != -INFINITY) {
        for (int s = 0; s < P.kv_splits; ++s) {
            const float ls = P.part_lse[s * split_l + li];
            const float w = ls == -INFINITY ? 0.0f : ex2(ls - M);
            wsum += w;
            const uint4 v = *reinterpret_cast<const uint4 *>(P.part_o + s * split_o + (size_t)r * D + c8);
            const uint32_t vs[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&vs[k]));
                acc[2 * k] = fmaf(w, f.x, acc[2 * k]);
                acc[2 * k + 1] = fmaf(w, f.y, acc[2 * k + 1]);
            }
        }
    }
    const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
    uint32_t w4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w4[k] = pack_bf16(acc[2 * k] * inv, acc[2 * k + 1] * inv);
    *reinterpret_cast<uint4 *>(P.out + (size_t)r * D + c8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
}

template <int D, bool CACHED>
cudaError_t run_attn(const AttentionProblem &p, unsigned *err, cudaStream_t stream)
{
    using L = ASmem<D>;
    const int G = p.Hq / p.Hkv;
    const int R = kRows / G;
    CUtensorMap tq, tk, tv;
    // Q viewed as [B*Hq, S, D]; box {64, R, G}: the G heads of one group, R positions each
    const uint64_t dq[3] = {(uint64_t)D, (uint64_t)p.S, (uint64_t)p.B * p.Hq};
    const uint64_t sq[2] = {(uint64_t)D * 2, (uint64_t)p.S * D * 2};
    const uint32_t bq[3] = {64, (uint32_t)R, (uint32_t)G};
    // K, V viewed as [B*Hkv, kv_seq, D] (16-bit elements; the copy is type-blind)
    const uint64_t dk[3] = {(uint64_t)D, (uint64_t)p.kv_seq, (uint64_t)p.B * p.Hkv};
    const uint64_t sk[2] = {(uint64_t)D * 2, (uint64_t)p.kv_seq * D * 2};
    const uint32_t bk[3] = {64, (uint32_t)kKeys, 1};
    if (encode_tmap(&tq, p.q, 3, dq, sq, bq, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tk, p.k, 3, dk, sk, bk, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tv, p.v, 3, dk, sk, bk, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    AttnParams a{};
    a.B = p.B;
    a.S = p.S;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.G = G;
    a.R = R;
    a.n_qblk = (p.S + kTiles * R - 1) / (kTiles * R);
    a.causal = p.causal;
    a.kv_splits = (CACHED && p.kv_splits > 1 && p.part_o && p.part_lse) ? p.kv_splits : 1;  // the cached variant only
    a.part_o = p.part_o;
    a.part_lse = p.part_lse;
    a.num_items = p.B * p.Hkv * a.n_qblk * a.kv_splits;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    a.kv_seq = p.kv_seq;
    a.kv_start = p.kv_start;
    a.out = p.out;
    a.lse = p.lse;
    a.lse_ld = p.lse_ld;
    a.err = err;
    auto kern = attn_kernel<D, CACHED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    {
        LaunchCfg lc(dim3(a.num_items), dim3(kThreads), L::ALLOC, stream, p.pdl != 0);
        e = cudaLaunchKernelEx(&lc.cfg, kern, tq, tk, tv, a);
        if (e != cudaSuccess) return e;
    }
    if (a.kv_splits > 1) {  // merge the key splits, as the attention kernel's programmatic dependent
        const int rows = p.B * p.S * p.Hq;
        const long long threads = (long long)rows * (D / 8);
        LaunchCfg lc(dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, stream, true);
        e = cudaLaunchKernelEx(&lc.cfg, combine_kernel<D>, a, rows);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttentionProblem &p, unsigned *err, int num_sms, cudaStream_t stream)
{
    (void)num_sms;
    if (p.d == 256) return launch_attention256(p, err, stream);
    if (p.Hkv <= 0 || p.Hq % p.Hkv) return cudaErrorInvalidValue;
    const int G = p.Hq / p.Hkv;
    if (G > kRows) return cudaErrorInvalidValue;
    if (p.cached) {
        if (p.d == 128) return run_attn<128, true>(p, err, stream);
        if (p.d == 64) return run_attn<64, true>(p, err, stream);
        if (p.d == 80) return run_attn<80, true>(p, err, stream);
        if (p.d == 96) return run_attn<96, true>(p, err, stream);
    } else {
        if (p.d == 128) return run_attn<128, false>(p, err, stream);
        if (p.d == 64) return run_attn<64, false>(p, err, stream);
        if (p.d == 80) return run_attn<80, false>(p, err, stream);
        if (p.d == 96) return run_attn<96, false>(p, err, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gqa

// prefill_umma.cuh -- paged prefill / chunked prefill attention on the tcgen05 tensor cores (fp16 /
// bf16), accumulators in tensor memory.
//
// A chunk of n new tokens per sequence attends causally to the sequence's cache through its block
// table ("PagedAttention e continuous batching", "01 - Conceito", paragraph 5: long prompts are
// sliced into chunks; "04 - Hacia PagedAttention (vista previa)", "La idea de PagedAttention",
// step 5: the kernel gathers the rows itself). The chunk's tokens are the newest, already
// appended: with c = context_lens[s] they sit at positions c - n .. c - 1, and position p sees keys
// 0 .. p. Unlike decode this is a dense contraction (n query rows x c keys x head_dim).
//
// CTA = (128 query rows, KV head, sequence); rows = token x head-in-group (GQA rows packed, so each
// K/V tile serves all G heads). Tiles are BN = 128 keys (eight 16-token blocks), so S = Q K^T runs as
// N = 128 instructions: ~64 cycles each on the tensor pipe, against ~50 cycles for one thread to
// issue one (an N = 64 instruction would leave the pipe waiting for its issuer). Eight warps:
//   warps 0-3  softmax: thread t owns query row t, which is TMEM lane t (a warp reaches only its
//              own 32 lanes). It first writes its row of Q into TMEM (the A operand of S = Q K^T:
//              no shared-memory reads of Q per instruction; the warp loads its 32 rows coalesced
//              and turns them around through shared memory), then per tile reads its row of S,
//              masks by selection, keeps the running max and sum in registers and writes its row
//              of P (storage type) into TMEM (d <= 128) or shared memory (d = 256, where TMEM is
//              full: S 128 + O 256 + Q 128 columns); at the end it scales its row of O by 1 / sum
//              and the warp stores its rows coalesced, staged in the idle K ring;
//   warps 4, 6 producers: walk the block table and move the K tiles (warp 4; a 2-D copy per block
//              and 64-column panel, landing panel-major so that S = Q K^T reads 128 keys per
//              instruction) and V stages of VB blocks (warp 6; one 3-D copy per block, landing
//              block-major: a PV instruction reads one 16-key block) into rings of STK / STV
//              stages (128-byte swizzle); a K stage is released when S_j is done, a V stage when
//              the PV instructions that read it are; warp 6 zeroes the V rows of skipped blocks
//              and of the positions past the context;
//   warp 5     S issuer (one thread): S_j = Q K_j^T into one of SB TMEM buffers (128 x BN fp32),
//              then a tcgen05.commit onto an mbarrier;
//   warp 7     PV issuer (one thread): O += P_j V_j into a TMEM accumulator (128 x D fp32, one
//              N = D instruction per 16 keys), V stage by V stage, each followed by commits that
//              free that part of P and that V stage. Two issuers keep the pipe fed while each
//              waits on its own barriers.
// S_{j+1} runs on the tensor pipe while the softmax warps work on S_j (they read S_j into registers
// first and release its buffer).
// At head_dim 256 two CTAs (a cluster of two adjacent query tiles) compute as one pair with
// .cta_group::2 instructions (M = 256 rows, 128 per CTA): each CTA loads half of every K tile and
// half of every V block, the even CTA issues the products, and the two exchange barrier arrivals
// (see the kernel's comment); the roles of the warps are otherwise the same.
// O is rescaled (read, multiplied, written back in TMEM) only when a row's running maximum grows
// by more than 8 (a factor 2^8 in the weights): P <= 2^8 stays exact enough in the storage type
// and the final division by the same running sum keeps the result the softmax's. The weights are
// 2^(s * scale * log2 e - m) from one FFMA and one ex2.approx each; the running sum adds them in
// fp32 before they are rounded to the storage type for the PV product.
// Each mbarrier serves one buffer, and no thread waits on a phase two completions old, so phase
// parities never alias. Every wait is bounded (PKV_DEV_WAIT_TIMEOUT).
#pragma once

#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "decode_mma.cuh"
#include "internal.h"
#include "umma.cuh"

namespace pkv {

// 2-D tensor copy of a 64-column x 16-row box with the default L2 policy (the K/V tiles of a prefill
// are re-read by every query tile of the sequence, so they should stay in L2).
__device__ __forceinline__ void tma_load_2d_keep(uint32_t dst, const void* tmap, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// 3-D tensor copy of the panels pan0 .. of one (block, KV head) chunk: box 64 columns x 16 rows x
// the map's panel count (all D/64 panels, or half of them for a CTA pair), landing as
// [panel][16 rows][128 B] (tensor maps of the PKV_BOX_BLOCK / PKV_BOX_BLOCK_HALF kinds).
__device__ __forceinline__ void tma_load_3d_keep(uint32_t dst, const void* tmap, int row, int pan0, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(0), "r"(row), "r"(pan0), "r"(smem_addr(bar))
        : "memory");
}

// 2^x with the ex2.approx.ftz instruction (2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed pairs of fp32 (the .f32x2 instructions of sm_100-family parts: two lanes of work per issue).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Weights of one row of a tile: p = 2^(s * sl - msub) (ex2.approx; a masked score, -inf, gives
// exactly 0), packed to the storage type in pw, their fp32 sums accumulated in ls (8 partial sums).
// The scale-and-subtract and the sums run as .f32x2 instructions: the softmax thread is bound by
// instruction issue (one warp per sub-partition), not by the ex2 unit — moving 7 of every 16 pairs
// onto an FMA-pipe polynomial made the kernel 11 % slower, packing these two steps 4 % faster.
template <typename M, int BN>
__device__ __forceinline__ void softmax_weights(const float (&sc)[BN], float sl, float msub, uint32_t (&pw)[BN / 2],
                                                float (&ls)[8]) {
    const uint64_t sl2 = f2_pack(sl, sl);
    const uint64_t nm2 = f2_pack(-msub, -msub);
    uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int c = 0; c < BN / 2; ++c) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(sc[2 * c], sc[2 * c + 1]), sl2, nm2), x0, x1);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        pw[c] = M::pack(p0, p1);
        ls2[c & 3] = f2_add(ls2[c & 3], f2_pack(p0, p1));
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) f2_unpack(ls2[c], ls[2 * c], ls[2 * c + 1]);
}

template <int D>
struct UmmaTuning {
    // Keys per tile: 128, so that S = Q K^T runs as N = 128 instructions (one issuing thread cannot
    // keep up with N = 64 instructions).
    static constexpr int BN = 128;
    // head_dim 256: CTA pairs. Alone, a CTA's shared memory carries ~320 KiB per 128-key tile (TMA
    // writes of K and V, tensor-core reads of K, V and P, the softmax's writes of P): ~2,560 cycles
    // at 128 B/cycle against 2,048 cycles of tensor work. Paired (a cluster of two CTAs holding
    // adjacent query tiles of one sequence and KV head, .cta_group::2 instructions with M = 256),
    // each CTA holds half of every K tile (64 of its 128 keys) and half of every V block (128 of
    // the 256 columns): ~192 KiB per tile per SM, and half the L2 -> SM traffic.
    static constexpr bool PAIR = D == 256;
    static constexpr bool PT = D <= 128;          // P in TMEM (A operand of PV) rather than shared memory
    static constexpr int SB = D == 256 ? 1 : 2;    // S buffers in TMEM
    static constexpr int STK = D == 256 ? 3 : (D == 128 ? 3 : 4);  // K stages
    // V stages hold VB 16-key blocks each, block-major ([block][panel][16 rows][128 B], one 3-D TMA
    // copy per block): half-tile stages at d = 256, so V of tile j+1 streams in while PV_j still
    // reads the other half.
    static constexpr int VB = D == 256 ? 4 : 8;
    static constexpr int STV = D == 256 ? 4 : (D == 128 ? 3 : 4);  // V stages
    static constexpr int NP = D == 64 ? 2 : 1;     // P buffers
    // TMEM columns: S [0, SB*BN), O [SB*BN, +D), Q [.., +D/2), P [.., +NP*BN/2) when PT (16-bit
    // operands hold two elements per 32-bit column)
    static constexpr uint32_t S_COL = 0, O_COL = SB * BN, Q_COL = SB * BN + D, P_COL = Q_COL + D / 2;
    static constexpr uint32_t USED = P_COL + (PT ? NP * BN / 2 : 0);
    static constexpr uint32_t TMEM_COLS = USED <= 256 ? 256u : 512u;
    static_assert(USED <= 512, "tensor memory");
};

template <int D>
struct UmmaSmem {
    using Tu = UmmaTuning<D>;
    static constexpr int BN = Tu::BN;
    static constexpr int KH = Tu::PAIR ? BN / 2 : BN;   // keys of each K tile this CTA holds
    static constexpr int DH = Tu::PAIR ? D / 2 : D;     // V columns this CTA holds
    static constexpr size_t KT = (size_t)KH * D * 2;    // K tile [D/64][KH keys][128 B]
    static constexpr size_t VT = (size_t)Tu::VB * 16 * DH * 2;  // V stage [VB][DH/64][16 keys][128 B]
    static constexpr size_t PB = Tu::PT ? 0 : (size_t)128 * BN * 2;  // P [BN/64][128 rows][128 B]
    static constexpr size_t K = 0;                       // [STK] K tiles
    static constexpr size_t V = K + (size_t)Tu::STK * KT;  // [STV] V stages
    static constexpr size_t P = V + (size_t)Tu::STV * VT;  // [NP] P tiles
    // Q staging at the start, QC columns of all 128 rows per pass (16-byte units of a row XOR-swizzled
    // by the row): the P buffer where P lives in shared memory (first written after every softmax
    // thread has moved its row of Q into tensor memory), else a region of its own
    static constexpr int QC = D < 128 ? D : 128;
    static constexpr size_t QSB = (size_t)128 * QC * 2;
    static constexpr bool Q_IN_P = Tu::NP * PB >= QSB;
    static constexpr size_t QS = Q_IN_P ? P : P + (size_t)Tu::NP * PB;
    static constexpr size_t BARS = Q_IN_P ? P + (size_t)Tu::NP * PB : QS + QSB;
    // full_k[STK] k_empty[STK] full_v[STV] v_empty[STV] s_full[SB] s_free[SB] p_full[NP * VPT]
    // p_free[NP * VPT] (one pair per part of a P buffer that one V stage's instructions read)
    // vtail q_ready
    static constexpr int NPP = Tu::NP * (Tu::BN / 16 / Tu::VB);
    static constexpr int NBARS = 2 * Tu::STK + 2 * Tu::STV + 2 * Tu::SB + 2 * NPP + 2;
    static constexpr size_t TADDR = BARS + (size_t)NBARS * 8;  // TMEM base address
    // output staging at the end (in the K ring): 128 rows of D * 2 bytes, 16 bytes apart in banks
    static constexpr size_t OROW = (size_t)D * 2 + 16;
    static_assert(128 * OROW <= (size_t)Tu::STK * KT, "output rows fit in the K ring");
    static constexpr size_t TOTAL = TADDR + 16;
    static constexpr size_t ALLOC = TOTAL + 1024;
};

// Paired CTAs (head_dim 256) split the work of one 256-row product as follows; the even CTA of the
// cluster ("lead") issues every tcgen05.mma, the odd one ("peer") supplies half of the operands
// and reads its half of the results from its own tensor memory:
//   - both load their half of each K tile / V stage with their own tensor copies onto their own
//     full_k / full_v barrier; the peer's warp 5 (K) and warp 7 (V) forward each completed phase
//     to the lead's barrier, which therefore counts two arrivals (its own expect_tx and the peer's);
//   - the peer's softmax threads arrive on the lead's q_ready, s_free and p_full barriers and its V
//     producer on the lead's vtail (each count doubled);
//   - the lead's MMA completions (commits onto its own s_full / k_empty and p_free / v_empty) are
//     forwarded to the peer's barriers of the same name by the thread that issued them, once they
//     have completed: S_{j+1} cannot start before both CTAs have read S_j (one S buffer), nor
//     PV_{j+1} before both have rewritten P (one P buffer), so the issuer would wait there anyway.
//     (A completion signal sent to both CTAs by the commit itself measured the same: the paired
//     kernel runs at the part's power limit.)
// A forwarded phase cannot be overtaken by the next one: every next phase of these barriers needs
// an arrival that depends on the forwarded one. Every wait is bounded, and a CTA that gives up
// still meets the other at the cluster barrier before it leaves. Remote arrivals carry the
// instruction's default (CTA-scope) semantics: a cluster-scope release put microseconds on every
// hand-off.
template <typename T, int D, int G>
__global__ void __launch_bounds__(256, 1)
    paged_prefill_umma_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v) {
    static_assert(128 % G == 0, "whole tokens per tile");
    using Tu = UmmaTuning<D>;
    using S = UmmaSmem<D>;
    using M = MmaType<T>;
    constexpr bool PAIR = Tu::PAIR;
    constexpr int CG = PAIR ? 2 : 1;
    constexpr int BN = Tu::BN, SB = Tu::SB, STK = Tu::STK, STV = Tu::STV, NP = Tu::NP;
    constexpr int BPT = BN / kBlock;                    // blocks per tile
    constexpr int KB = S::KH / kBlock;                  // blocks of each K tile this CTA loads
    constexpr int ROWS = 128;
    constexpr int QT = ROWS / G;
    constexpr int PANELS = D / 64;                      // panels of a K block
    constexpr int VPAN = S::DH / 64;                    // panels of a V block in this CTA
    constexpr uint32_t KT = (uint32_t)S::KT;
    constexpr uint32_t VT = (uint32_t)S::VT;
    constexpr uint32_t PANEL = S::KH * 128;             // one 64-column panel of this CTA's K tile
    constexpr uint32_t KBLKB = kBlock * D * 2;          // one K block (all panels)
    constexpr uint32_t BLKB = kBlock * S::DH * 2;       // this CTA's part of one V block
    constexpr int VB = Tu::VB;
    constexpr int VPT = BPT / VB;                       // V stages per tile
    static_assert(BPT % VB == 0, "whole V stages per tile");
    static_assert(Tu::PT ? VPT == 1 : (VB * kBlock) % 64 == 0, "a P part is whole 64-key panels");
    constexpr bool BF = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t IDESC_S = umma_idesc_f16(BF, PAIR ? 256 : 128, BN, false);
    constexpr uint32_t IDESC_PV = umma_idesc_f16(BF, PAIR ? 256 : 128, D, true);
    constexpr uint32_t S_COL = Tu::S_COL, O_COL = Tu::O_COL, Q_COL = Tu::Q_COL;
    static_assert(BPT <= 32, "one lane per block of a tile");

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint64_t* full_k = reinterpret_cast<uint64_t*>(smem + S::BARS);
    uint64_t* k_empty = full_k + STK;
    uint64_t* full_v = k_empty + STK;
    uint64_t* v_empty = full_v + STV;
    uint64_t* s_full = v_empty + STV;
    uint64_t* s_free = s_full + SB;
    uint64_t* p_full = s_free + SB;
    uint64_t* p_free = p_full + S::NPP;
    uint64_t* vtail = p_free + S::NPP;
    uint64_t* q_ready = vtail + 1;
    uint32_t* taddr_s = reinterpret_cast<uint32_t*>(smem + S::TADDR);
    const uint32_t sbase = smem_addr(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // A launch that follows this one as a programmatic dependent (the next layer's attention of
    // the same chunk) may start once every CTA has passed here and fill the SMs this grid's last
    // wave leaves idle. Without such a launch this is a no-op.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool lead = rank == 0;
    const int tile = a.q_tiles - 1 - (int)blockIdx.x;  // tiles with the most keys start first
    const int g = blockIdx.y;
    const int s = blockIdx.z;

    const int q0 = a.q_start[s];
    const int q1 = a.q_start[s + 1];
    const int n_new = q1 - q0;
    const int ctx = a.lens[s];
    const bool bad = q0 < 0 || q1 > a.n_tokens || n_new < 0 || n_new > a.q_tiles * QT || ctx < n_new ||
                     ctx > a.max_blocks * kBlock;
    if (bad && blockIdx.x == 0 && g == 0 && threadIdx.x == 0) atomicOr(a.status, (unsigned)PKV_DEV_BAD_QUERY_RANGE);
    // BN-key tiles a query tile needs: keys 0 .. the position of its last token (0: no rows)
    auto key_tiles = [&](int qt) -> int {
        const int tq0 = qt * QT;
        if (bad || qt < 0 || tq0 >= n_new) return 0;
        return (ctx - n_new + min(tq0 + QT, n_new) - 1) / BN + 1;
    };
    // A pair walks the key tiles of its heavier query tile: both CTAs take part in every product
    // (the lighter tile's causal mask zeroes the keys it does not see). Both compute the same count.
    int n_tiles = key_tiles(tile);
    if constexpr (PAIR) n_tiles = max(n_tiles, key_tiles(a.q_tiles - 1 - (int)(blockIdx.x ^ 1u)));
    if (n_tiles == 0) return;  // both CTAs of a pair leave here together, before any cluster barrier
    const int t0 = tile * QT;
    const int pos0 = ctx - n_new + t0;
    const int nb = (ctx + kBlock - 1) / kBlock;
    const bool tail_tile = n_tiles * BN > ctx;  // the last tile holds rows past the context
    // The tile's query rows, loaded here by the softmax warps with every load in flight at once, so
    // that their latency overlaps the barrier and tensor-memory setup below. Coalesced: a load
    // instruction covers RPI rows' QC-column segments (LPR lanes of 16 bytes each per row), and the
    // softmax role turns the warp's 32 rows around through shared memory so that thread t holds row t
    // (TMEM lane t). (One row per thread straight from global memory cost each CTA ~2.5-4 us: every
    // 16-byte load of a warp touched 32 rows.)
    constexpr int QC = S::QC;
    constexpr int QPASS = D / QC;        // passes of QC columns
    constexpr int LPR = QC * 2 / 16;     // lanes per row segment (16 or 8)
    constexpr int RPI = 32 / LPR;        // rows per load instruction
    constexpr int QI = 32 / RPI;         // load instructions per pass
    static_assert(LPR % 8 == 0 && LPR <= 16, "a row segment spans whole 128-byte bank sets");
    uint4 qreg[QPASS * QI];
    if (threadIdx.x < ROWS) {
        const int l = threadIdx.x & 31;
#pragma unroll
        for (int i = 0; i < QI; ++i) {
            const int r = (threadIdx.x & ~31) + i * RPI + l / LPR;  // query row of this load
            const int tt = r / G;
            const bool live = t0 + tt < n_new;
            const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.q) +
                                                              ((size_t)(q0 + t0 + tt) * a.n_q + (size_t)g * G + r % G) * D) +
                               l % LPR;
#pragma unroll
            for (int pass = 0; pass < QPASS; ++pass)
                qreg[pass * QI + i] = live ? __ldg(src + pass * (QC / 8)) : make_uint4(0u, 0u, 0u, 0u);
        }
    }

    if (threadIdx.x == 0) {
        // the lead's barriers that the peer also arrives on count both CTAs' arrivals
        const uint32_t two = PAIR && lead ? 2u : 1u;
        for (int i = 0; i < STK; ++i) {
            mbar_init(&full_k[i], two);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < STV; ++i) {
            mbar_init(&full_v[i], two);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < SB; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 128 * two);
        }
        for (int i = 0; i < S::NPP; ++i) {
            mbar_init(&p_full[i], 128 * two);
            mbar_init(&p_free[i], 1);
        }
        mbar_init(vtail, 32 * two);
        mbar_init(q_ready, 128 * two);
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc_cg<CG>(taddr_s, Tu::TMEM_COLS);
    tcgen05_before_sync();
    __syncthreads();
    if constexpr (PAIR) cluster_sync_all();  // both CTAs' barriers and tensor memory exist from here on
    tcgen05_after_sync();
    const uint32_t tmem = *taddr_s;
    // an arrival on the lead's copy of one of this CTA's barriers (the peer's softmax threads and V
    // producer: one remote operation per warp that counts its lanes), or on this CTA's own when it is
    // the lead or works alone
    auto arrive_lead = [&](uint64_t* bar) {
        if (PAIR && !lead)
            mbar_arrive_remote_warp(cluster_addr(bar, 0u));
        else
            mbar_arrive(bar);
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool { return mbar_wait_bounded(bar, parity); };

    if (warp == 4 || warp == 6) {
        // ===================== producers: warp 4 moves K tiles, warp 6 moves V stages =====================
        // A K stage (one tile) is released once S_j has been computed, a V stage (VB blocks) once the
        // PV instructions that read it have: the next K tile lands while the softmax of this one runs.
        // Unit u: K tile u (its KB blocks of this CTA, panel-major, one 2-D copy per block and panel),
        // or V stage u (VB blocks of tile u / VPT, block-major, one 3-D copy per block of this CTA's
        // columns).
        const bool is_v = warp == 6;
        const int nst = is_v ? STV : STK;
        const int upt = is_v ? VPT : 1;           // units per tile
        const int nbu = is_v ? VB : KB;           // blocks per unit this CTA loads
        const int n_units = n_tiles * upt;
        uint64_t* full = is_v ? full_v : full_k;
        uint64_t* empty = is_v ? v_empty : k_empty;
        const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
        const uint32_t ring = (uint32_t)(is_v ? S::V : S::K);
        const uint32_t ust = is_v ? VT : KT;      // bytes per stage
        const uint32_t ubb = is_v ? BLKB : KBLKB; // bytes per block this CTA copies
        // first block of unit u this CTA loads: V stages tile the block list; a pair splits each
        // K tile's blocks between its CTAs (the lead the first KB)
        auto unit_block0 = [&](int u) -> int { return is_v ? u * VB : u * BPT + (int)rank * KB; };
        const int32_t* trow = a.tables + (size_t)s * a.max_blocks;
        int issued = 0;
        // lane l < nbu handles block l of every unit; its table entry is read one unit ahead, so
        // that the load's latency overlaps the wait for a free stage
        int phys_next = lane < nbu && unit_block0(0) + lane < nb ? __ldg(trow + unit_block0(0) + lane) : -1;
        for (int u = 0; u < n_units; ++u) {
            const int j = u / upt;
            const int st = u % nst;
            const int blk = unit_block0(u) + lane;
            const bool inb = lane < nbu && blk < nb;
            const int phys = phys_next;
            const int nblk = unit_block0(u + 1) + lane;
            phys_next = lane < nbu && nblk < nb ? __ldg(trow + nblk) : -1;
            if (u >= nst && !wait(&empty[st], (uint32_t)((u / nst) - 1) & 1u)) {
                if (lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
                break;
            }
            const bool ok = inb && (unsigned)phys < (unsigned)a.num_blocks;
            const unsigned okm = __ballot_sync(0xffffffffu, ok);
            const unsigned badm = __ballot_sync(0xffffffffu, inb && !ok);
            unsigned char* unit_ptr = smem + ring + (size_t)st * ust;
            if (badm) {
                // skipped blocks: keys masked by the softmax, V rows zeroed (P = 0 there, 0 * NaN is not)
                if (!is_v && lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_BAD_BLOCK_ID);
                if (is_v) {
                    for (int b = 0; b < VB; ++b) {
                        if (!((badm >> b) & 1u)) continue;
                        for (int i = lane; i < (int)(BLKB / 16); i += 32)
                            reinterpret_cast<uint4*>(unit_ptr + (size_t)b * BLKB)[i] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
            }
            if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)__popc(okm) * ubb);
            __syncwarp();
            if (ok) {
                const int row0 = (phys * a.n_kv + g) * kBlock;
                if (is_v) {
                    // this CTA's VPAN panels of the block: panels rank * VPAN .. of the row
                    tma_load_3d_keep(sbase + ring + (uint32_t)st * VT + (uint32_t)lane * BLKB, tm, row0,
                                     (int)rank * VPAN, &full[st]);
                } else {
                    const uint32_t dst = sbase + ring + (uint32_t)st * KT + (uint32_t)lane * 2048;
#pragma unroll
                    for (int pn = 0; pn < PANELS; ++pn) tma_load_2d_keep(dst + pn * PANEL, tm, pn * 64, row0, &full[st]);
                }
            }
            issued = u + 1;
            if (is_v && j == n_tiles - 1 && tail_tile) {
                // zero this stage's rows past the context (key rows r0 .. BN-1 of the last tile)
                if (!mbar_wait_bounded(&full_v[st], (uint32_t)(u / nst) & 1u)) {
                    if (lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
                    break;
                }
                const int r0 = ctx - j * BN;               // 1 .. BN-1
                const int lo = max(r0 - (u % VPT) * VB * kBlock, 0);  // first stage row to zero
                for (int i = lane; i < (VB * kBlock - lo) * VPAN * 8; i += 32) {
                    const int r = lo + i / (VPAN * 8);    // stage row = 16 x block + token
                    const int pn = (i / 8) % VPAN;
                    reinterpret_cast<uint4*>(unit_ptr + (size_t)(r / kBlock) * BLKB + (size_t)pn * 2048 +
                                             (size_t)(r % kBlock) * 128)[i % 8] = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                if (u == n_units - 1) arrive_lead(vtail);
            }
        }
        for (int u = max(0, issued - nst); u < issued; ++u)  // the copies of the last stages have landed
            mbar_wait_bounded(&full[u % nst], (uint32_t)(u / nst) & 1u);
    } else if (PAIR && !lead && (warp == 5 || warp == 7)) {
        // ===================== peer: forward this CTA's landed K tiles (warp 5) and V stages (warp 7) =====================
        if (lane == 0) {
            const bool is_v = warp == 7;
            const int nst = is_v ? STV : STK;
            const int n_units = n_tiles * (is_v ? VPT : 1);
            uint64_t* full = is_v ? full_v : full_k;
            for (int u = 0; u < n_units; ++u) {
                if (!mbar_wait_bounded(&full[u % nst], (uint32_t)(u / nst) & 1u)) {
                    atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
                    break;
                }
                mbar_arrive_remote(cluster_addr(&full[u % nst], 0u));
            }
        }
        __syncwarp();
    } else if (warp == 5 || warp == 7) {
        // ===================== MMA issuers: warp 5 S = Q K^T, warp 7 O += P V =====================
        // Two issuing threads: a tcgen05.mma takes ~50 cycles to issue from one thread and an
        // N = 128 instruction ~64 cycles on the tensor pipe, so one thread interleaving both products
        // and their barrier waits would leave the pipe idle. Descriptors are built once per stage
        // and stepped by constant offsets (shared-memory addresses stay below 2^18 bytes, so the
        // 14-bit address field never carries).
        if (lane == 0) {
            bool ok = true;
            if (warp == 5) {
                const uint64_t kdesc0 = umma_desc_sw128(sbase + (uint32_t)S::K, 16, 1024);
                ok = wait(q_ready, 0u);
                for (int j = 0; ok && j < n_tiles; ++j) {
                    const int st = j % STK;
                    const int b = j % SB;
                    if (!wait(&full_k[st], (uint32_t)(j / STK) & 1u) ||
                        (j >= SB && !wait(&s_free[b], (uint32_t)((j / SB) - 1) & 1u))) {
                        ok = false;
                        break;
                    }
                    tcgen05_after_sync();
                    const uint64_t kd = kdesc0 + (uint64_t)(((uint32_t)st * KT) >> 4);
                    const uint32_t d_s = tmem + S_COL + (uint32_t)(b * BN);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        umma_f16_tmem_a_cg<CG>(d_s, tmem + Q_COL + (uint32_t)ks * 8,
                                               kd + (uint64_t)(((uint32_t)(ks >> 2) * PANEL + (uint32_t)(ks & 3) * 32) >> 4),
                                               IDESC_S, ks > 0);
                    umma_commit_cg<CG>(&s_full[b]);
                    umma_commit_cg<CG>(&k_empty[st]);  // the K stage may take tile j + STK once S_j is done
                    if constexpr (PAIR) {
                        // S_j done: the peer may read its rows of S_j and refill its half of the K stage
                        if (!mbar_wait_bounded(&s_full[b], (uint32_t)(j / SB) & 1u) ||
                            !mbar_wait_bounded(&k_empty[st], (uint32_t)(j / STK) & 1u)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_remote(cluster_addr(&s_full[b], 1u));
                        mbar_arrive_remote(cluster_addr(&k_empty[st], 1u));
                    }
                }
            } else {
                // V stage: block kk of the tile at + (kk % VB) * BLKB, its panels 2 KiB apart (leading
                // byte offset), 8-key core groups 1 KiB apart (stride byte offset)
                const uint64_t vdesc0 = umma_desc_sw128(sbase + (uint32_t)S::V, 2048, 1024);
                const uint64_t pdesc0 = umma_desc_sw128(sbase + (uint32_t)S::P, 16, 1024);
                for (int j = 0; ok && j < n_tiles; ++j) {
                    const int pb = j % NP;
                    if (j == n_tiles - 1 && tail_tile && !wait(vtail, 0u)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int h = 0; h < VPT; ++h) {
                        // part h of P_j (the keys of V stage u) and the V stage itself
                        const int u = j * VPT + h;
                        const int sv = u % STV;
                        if (!wait(&p_full[pb * VPT + h], (uint32_t)(j / NP) & 1u) ||
                            !wait(&full_v[sv], (uint32_t)(u / STV) & 1u)) {
                            ok = false;
                            break;
                        }
                        tcgen05_after_sync();
                        const uint64_t vd = vdesc0 + (uint64_t)(((uint32_t)sv * VT) >> 4);
#pragma unroll
                        for (int i = 0; i < VB; ++i) {
                            const int kk = h * VB + i;
                            const uint64_t bd = vd + (uint64_t)(((uint32_t)i * BLKB) >> 4);
                            if constexpr (Tu::PT) {
                                umma_f16_tmem_a_cg<CG>(tmem + O_COL, tmem + Tu::P_COL + (uint32_t)(pb * (BN / 2) + kk * 8),
                                                       bd, IDESC_PV, j > 0 || kk > 0);
                            } else {
                                const uint64_t ad = pdesc0 + (uint64_t)(((uint32_t)pb * (uint32_t)S::PB +
                                                                         (uint32_t)(kk >> 2) * (128 * 128) +
                                                                         (uint32_t)(kk & 3) * 32) >> 4);
                                umma_f16_cg<CG>(tmem + O_COL, ad, bd, IDESC_PV, j > 0 || kk > 0);
                            }
                        }
                        umma_commit_cg<CG>(&p_free[pb * VPT + h]);  // part h of P buffer pb may take P_{j+NP}
                        umma_commit_cg<CG>(&v_empty[sv]);           // the V stage may take unit u + STV
                    }
                    if constexpr (PAIR) {
                        // PV_j done part by part: the peer may rewrite that part of its P and refill
                        // its half of the V stage
#pragma unroll
                        for (int h = 0; ok && h < VPT; ++h) {
                            const int u = j * VPT + h;
                            if (!mbar_wait_bounded(&p_free[pb * VPT + h], (uint32_t)(j / NP) & 1u) ||
                                !mbar_wait_bounded(&v_empty[u % STV], (uint32_t)(u / STV) & 1u)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_remote(cluster_addr(&p_free[pb * VPT + h], 1u));
                            mbar_arrive_remote(cluster_addr(&v_empty[u % STV], 1u));
                        }
                    }
                }
            }
            if (!ok) atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
            const int last = n_tiles - 1;
            // this thread's MMAs have completed before TMEM is released (its last commit covers them all)
            if (warp == 5)
                mbar_wait_bounded(&s_full[last % SB], (uint32_t)(last / SB) & 1u);
            else
                mbar_wait_bounded(&p_free[(last % NP) * VPT + VPT - 1], (uint32_t)(last / NP) & 1u);
        }
        __syncwarp();
    } else {
        // ===================== softmax (warps 0-3): thread = query row = TMEM lane =====================
        const int row = threadIdx.x;
        const int tt = row / G;
        const int lim = min(pos0 + tt, ctx - 1);
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const float sl = a.scale_log2;
        {
            // this thread's query row -> TMEM lane `row` (the A operand of S = Q K^T; zero past the
            // chunk): the warp's loaded segments go to its own 32 rows of the staging area, unit u of
            // row rr at 16-byte position u ^ (rr & 7) (eight consecutive rows in distinct banks), and
            // each thread reads its row back
            unsigned char* qs = smem + S::QS + (size_t)warp * 32 * (QC * 2);
#pragma unroll
            for (int pass = 0; pass < QPASS; ++pass) {
                if (pass > 0) __syncwarp();  // the previous pass has been read
#pragma unroll
                for (int i = 0; i < QI; ++i) {
                    const int rr = i * RPI + lane / LPR;
                    *reinterpret_cast<uint4*>(qs + (size_t)rr * (QC * 2) + (size_t)(((lane % LPR) ^ (rr & 7)) << 4)) =
                        qreg[pass * QI + i];
                }
                __syncwarp();
                uint32_t qv[QC / 2];
#pragma unroll
                for (int u = 0; u < LPR; ++u) {
                    const uint4 x =
                        *reinterpret_cast<const uint4*>(qs + (size_t)lane * (QC * 2) + (size_t)((u ^ (lane & 7)) << 4));
                    qv[4 * u] = x.x;
                    qv[4 * u + 1] = x.y;
                    qv[4 * u + 2] = x.z;
                    qv[4 * u + 3] = x.w;
                }
#pragma unroll
                for (int c0 = 0; c0 < QC / 2; c0 += 32)
                    tmem_st32(tmem + lane_base + Q_COL + (uint32_t)(pass * (QC / 2) + c0),
                              *reinterpret_cast<const uint32_t(*)[32]>(&qv[c0]));
            }
            tmem_wait_st();
            tcgen05_before_sync();
            arrive_lead(q_ready);
        }
        float m_used = -INFINITY;
        float l = 0.f;
        bool ok = true;
        // which of a tile's blocks were loaded (a table entry out of range is skipped): read from the
        // table itself one tile ahead, so that no wait on a producer's barrier is needed here
        const int32_t* trow = a.tables + (size_t)s * a.max_blocks;
        auto tile_mask = [&](int j) -> unsigned {
            unsigned m = 0;
#pragma unroll
            for (int bb = 0; bb < BPT; ++bb) {
                const int blk = j * BPT + bb;
                if (blk < nb && (unsigned)__ldg(trow + blk) < (unsigned)a.num_blocks) m |= 1u << bb;
            }
            return m;
        };
        constexpr unsigned FULL = (1u << BPT) - 1u;
        unsigned okm_next = tile_mask(0);
        for (int j = 0; j < n_tiles; ++j) {
            const int b = j % SB;
            const int pb = j % NP;
            const unsigned okm = okm_next;
            if (j + 1 < n_tiles) okm_next = tile_mask(j + 1);
            if (!wait(&s_full[b], (uint32_t)(j / SB) & 1u)) {
                ok = false;
                break;
            }
            tcgen05_after_sync();
            float sc[BN];
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 32)
                tmem_ld32(tmem + lane_base + S_COL + (uint32_t)(b * BN + c0), *reinterpret_cast<uint32_t(*)[32]>(&sc[c0]));
            tmem_wait_ld();
            tcgen05_before_sync();
            arrive_lead(&s_free[b]);  // the S buffer may take S_{j+SB}
            const int key0 = j * BN;
            const bool unmasked = key0 + BN - 1 <= lim && okm == FULL;
            if (!unmasked) {
#pragma unroll
                for (int c = 0; c < BN; ++c) {  // masking by selection: a masked score is -inf
                    const bool v = key0 + c <= lim && ((okm >> (c >> 4)) & 1u);
                    sc[c] = v ? sc[c] : -INFINITY;
                }
            }
            float mx4[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) mx4[c] = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN / 2; ++c) mx4[c & 3] = fmax3(mx4[c & 3], sc[2 * c], sc[2 * c + 1]);
            const float smax = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
            const float mt = smax * sl;  // the tile's row maximum in base 2 (scale > 0)
            // running maximum: move it (and rescale O, l) only when it grows by more than 8
            const bool grow = mt > m_used + 8.f;
            const float m_new = grow ? mt : m_used;
            const float alpha = grow ? exp2f(m_used - m_new) : 1.f;  // 0 when m_used is -inf
            if (j > 0 && __any_sync(0xffffffffu, grow)) {
                // O holds P_0..P_{j-1} V: wait for the last PV, then scale this warp's 32 rows in TMEM
                if (!wait(&p_free[((j - 1) % NP) * VPT + VPT - 1], (uint32_t)((j - 1) / NP) & 1u)) {
                    ok = false;
                    break;
                }
                tcgen05_after_sync();
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t ov[32];
                    tmem_ld32(tmem + lane_base + O_COL + (uint32_t)c0, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
                    tmem_st32(tmem + lane_base + O_COL + (uint32_t)c0, ov);
                }
                tmem_wait_st();
            }
            l *= alpha;
            m_used = m_new;
            // p = 2^(s * scale_log2 - m): one (packed) FFMA and one ex2 per score; a masked score
            // (-inf) gives exactly 0. While every score so far is masked m_used is -inf: subtract 0
            // instead.
            const float msub = m_used == -INFINITY ? 0.f : m_used;
            uint32_t pw[BN / 2];
            float lsf[8];
            softmax_weights<M>(sc, sl, msub, pw, lsf);
            l += ((lsf[0] + lsf[1]) + (lsf[2] + lsf[3])) + ((lsf[4] + lsf[5]) + (lsf[6] + lsf[7]));
            // part h of P buffer pb is free once the instructions of PV_{j-NP} that read it are done
#pragma unroll
            for (int h = 0; h < VPT; ++h) {
                if (j >= NP && !wait(&p_free[pb * VPT + h], (uint32_t)((j / NP) - 1) & 1u)) {
                    ok = false;
                    break;
                }
                if constexpr (Tu::PT) {
                    // this row of P -> TMEM lane `row`, two 16-bit weights per column
                    if (j >= NP) tcgen05_after_sync();
#pragma unroll
                    for (int c0 = 0; c0 < BN / 2; c0 += 32)
                        tmem_st32(tmem + lane_base + Tu::P_COL + (uint32_t)(pb * (BN / 2) + c0),
                                  *reinterpret_cast<const uint32_t(*)[32]>(&pw[c0]));
                    tmem_wait_st();
                } else {
                    unsigned char* prow = smem + S::P + (size_t)pb * S::PB + (size_t)row * 128;
#pragma unroll
                    for (int pp = h * (VB * kBlock / 64); pp < (h + 1) * (VB * kBlock / 64); ++pp)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4*>(prow + (size_t)pp * (128 * 128) + ((c ^ (row & 7)) << 4)) =
                                make_uint4(pw[32 * pp + 4 * c], pw[32 * pp + 4 * c + 1], pw[32 * pp + 4 * c + 2],
                                           pw[32 * pp + 4 * c + 3]);
                    fence_proxy_async_smem();
                }
                tcgen05_before_sync();
                arrive_lead(&p_full[pb * VPT + h]);
            }
            if (!ok) break;
        }
        if (ok) {
            const int last = n_tiles - 1;
            if (!wait(&p_free[(last % NP) * VPT + VPT - 1], (uint32_t)(last / NP) & 1u)) ok = false;
        }
        // launched as a programmatic dependent, this grid computed while the previous kernel was
        // finishing; the outputs are written only once that kernel has completed (so a chain of
        // such launches completes in order)
        grid_dependency_wait();
        if (!ok) {
            if (lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
        } else {
            tcgen05_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            // The rows go out through shared memory: written directly from the thread that owns a
            // row, every 16-byte store of a warp hit 32 rows (~2.4 us per CTA at head_dim 256). The K
            // ring is idle here: every K and V copy has landed and every product that read them has
            // completed (the last PV, which this thread has just waited for, follows them all). A
            // row stride of D * 2 + 16 bytes puts the 16-byte writes of eight consecutive rows in
            // distinct banks.
            unsigned char* srow = smem + S::K + (size_t)row * S::OROW;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 64) {
                uint32_t ov[64];
                tmem_ld32(tmem + lane_base + O_COL + (uint32_t)c0, *reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
                tmem_ld32(tmem + lane_base + O_COL + (uint32_t)c0 + 32u, *reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(srow + (size_t)c0 * 2 + 16 * c) =
                        make_uint4(M::pack(__uint_as_float(ov[8 * c]) * inv, __uint_as_float(ov[8 * c + 1]) * inv),
                                   M::pack(__uint_as_float(ov[8 * c + 2]) * inv, __uint_as_float(ov[8 * c + 3]) * inv),
                                   M::pack(__uint_as_float(ov[8 * c + 4]) * inv, __uint_as_float(ov[8 * c + 5]) * inv),
                                   M::pack(__uint_as_float(ov[8 * c + 6]) * inv, __uint_as_float(ov[8 * c + 7]) * inv));
            }
            __syncwarp();
            // then the warp's 32 rows leave UPR 16-byte units a row, RPS rows per store instruction
            // (512 contiguous bytes at head_dim 256); rows past the chunk are not written
            constexpr int UPR = D / 8;
            constexpr int RPS = 32 / UPR;
            const unsigned char* wrows = smem + S::K + (size_t)(warp * 32) * S::OROW;
#pragma unroll 4
            for (int k = 0; k < 32 / RPS; ++k) {
                const int rr = k * RPS + lane / UPR;
                const int r = warp * 32 + rr;
                const int t = r / G;
                if (t0 + t < n_new) {
                    T* dst = reinterpret_cast<T*>(a.out) + ((size_t)(q0 + t0 + t) * a.n_q + (size_t)g * G + r % G) * D;
                    reinterpret_cast<uint4*>(dst)[lane % UPR] =
                        *reinterpret_cast<const uint4*>(wrows + (size_t)rr * S::OROW + (size_t)(lane % UPR) * 16);
                }
            }
        }
    }
    tcgen05_before_sync();
    __syncthreads();
    // no CTA of a pair leaves (or releases its tensor memory) while the other may still arrive on
    // its barriers or the pair's products may still write its tensor memory
    if constexpr (PAIR) cluster_sync_all();
    if (warp == 5) {
        tcgen05_after_sync();
        tmem_dealloc_cg<CG>(tmem, Tu::TMEM_COLS);
    }
}

template <typename T, int D, int G>
cudaError_t launch_prefill_umma_tpl(const PrefillArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                    cudaStream_t stream) {
    using Tu = UmmaTuning<D>;
    constexpr size_t smem = UmmaSmem<D>::ALLOC;
    static_assert(smem <= 227 * 1024, "shared memory per CTA");
    auto kern = paged_prefill_umma_kernel<T, D, G>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    static unsigned long long attr_done = 0;
    if (dev < 64 && !(__atomic_load_n(&attr_done, __ATOMIC_ACQUIRE) & (1ull << dev))) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        __atomic_fetch_or(&attr_done, 1ull << dev, __ATOMIC_ACQ_REL);
    }
    constexpr int CL = Tu::PAIR ? 2 : 1;
    PrefillArgs b = a;
    b.q_tiles = (a.q_tiles + CL - 1) / CL * CL;  // whole pairs; an extra query tile has no rows
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(b.q_tiles, b.n_kv, b.n_seqs);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n_attr = 0;
    if (CL > 1) {
        attr[n_attr].id = cudaLaunchAttributeClusterDimension;
        attr[n_attr].val.clusterDim.x = CL;
        attr[n_attr].val.clusterDim.y = 1;
        attr[n_attr].val.clusterDim.z = 1;
        ++n_attr;
    }
    if (a.overlap_previous) {
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
        ++n_attr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    err = cudaLaunchKernelEx(&cfg, kern, b, tk, tv);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

// CTAs of the tensor-core prefill kernel the GPU holds at once (one wave): SMs x CTAs per SM (shared
// memory, registers, tensor memory), and for CTA pairs no more than the pairs the cluster scheduler
// can place at once (an SM without a free partner in its GPC cannot hold half a pair).
template <typename T, int D, int G>
cudaError_t prefill_umma_wave_ctas_tpl(int sms, int* out) {
    constexpr size_t smem = UmmaSmem<D>::ALLOC;
    auto kern = paged_prefill_umma_kernel<T, D, G>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem);
    if (err != cudaSuccess) return err;
    // tensor memory: a CTA allocates TMEM_COLS of the SM's 512 columns for its whole life
    const int by_tmem = 512 / (int)UmmaTuning<D>::TMEM_COLS;
    if (per_sm > by_tmem) per_sm = by_tmem;
    *out = sms * per_sm;
    if constexpr (UmmaTuning<D>::PAIR) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
        if (err != cudaSuccess) return err;
        if (2 * clusters < *out) *out = 2 * clusters;
    }
    return cudaSuccess;
}

template <typename T>
cudaError_t prefill_umma_wave_ctas_dtype(int head_dim, int group, int sms, int* out) {
#define PKV_CASE(DD, GG) \
    if (head_dim == DD && group == GG) return prefill_umma_wave_ctas_tpl<T, DD, GG>(sms, out);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
    PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_prefill_umma_dtype(int head_dim, int group, const PrefillArgs& a, const CUtensorMap& tk,
                                      const CUtensorMap& tv, cudaStream_t stream) {
#define PKV_CASE(DD, GG) \
    if (head_dim == DD && group == GG) return launch_prefill_umma_tpl<T, DD, GG>(a, tk, tv, stream);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
    PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv

// stream_decode.cu -- the decode expert block at S = 1 (one token, top-K routed
// experts) for int4 (fmt 2 and 4) and int8 (fmt 1) expert tables, in one
// cooperative launch with one CTA per SM (colibri-strix commit log, "metal:
// batched moe_block": gate/up GEMV, SiLU * mul, down GEMV and the weighted sum
// over the routed experts as a single GPU pass).
//
// Roles.  Warps 0 .. NC-1 (the consumers) form NG independent groups of GW
// warps.  Each group has SPG shared-memory slots of its own and its own stage
// sequence, fed by one lane of warp NC (the producer warp: lane g streams
// group g's weight rows into its slots with bulk copies, cp.async.bulk of
// whole rows and their group scales, and writes a descriptor per slot), so the
// groups run at their own pace.  Consumer lanes keep the activations of their
// 16-byte chunk of a row in registers as integer limbs (dp4a.cuh), so the dot
// product of a chunk is a few dp4a per word of codes.
//
//   phase 0: the token's routed experts, distinct and in ascending id order,
//            duplicate slots' weights summed.
//   phase A: stages of RP (gate, up) row pairs of one expert, dealt round
//            robin to the NG x gridDim groups of all CTAs.  A warp owns one 512-byte slab of
//            the rows; the last warp of the group to finish a stage sums the
//            slab partials of each pair in slab order and writes
//            h[a][j] = silu(g) * u to global scratch.
//   grid barrier among the consumers; the producer meanwhile copies the first
//            phase-B stages.
//   phase B: the CTA owns output rows [oc0, oc1).  Group g handles the routed
//            experts g, g + NG, ...; a phase-B stage holds RB rows of each of
//            them, and a warp owns one expert and SPW slabs of its rows, whose
//            h limbs it converts once, after the barrier.  y[o] = sum_a w_a *
//            sum_slabs d_a[o], summed in a fixed order, written once.
// Results do not depend on timing or on the number of SMs beyond f32
// reassociation inside a slab.  Every wait is bounded (mbarrier.cuh); on
// expiry the kernel records DEV_ERR_TIMEOUT and returns.  The last CTA to leave
// resets the call's barrier counter, whichever way the call ended.
#include <algorithm>
#include <cstring>

#include "coli_internal.cuh"
#include "decode_route.cuh"
#include "dp4a.cuh"
#include "mbarrier.cuh"

namespace coli {

namespace {

constexpr int kSdSlotsPerGroup = 2;   // a group streams into one slot while it consumes the other

// Stage descriptor, written by the producer into shared memory before it arms
// the stage's full barrier (the consumers read it after their wait).
enum : int { SD_A = 0, SD_B = 1, SD_END_A = 2, SD_END_B = 3 };

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ float ldsf(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// Sums of four per-lane values over the warp with 6 shuffles: afterwards lane
// 8k (k = 0..3) holds the total of value k.
__device__ __forceinline__ float sd_warp_sum4(float v0, float v1, float v2, float v3, int lane) {
    const bool h16 = lane & 16, h8 = lane & 8;
    float a0 = h16 ? v2 : v0, a1 = h16 ? v3 : v1;
    const float b0 = h16 ? v0 : v2, b1 = h16 ? v1 : v3;
    a0 += __shfl_xor_sync(0xffffffffu, b0, 16);
    a1 += __shfl_xor_sync(0xffffffffu, b1, 16);
    float k = h8 ? a1 : a0;
    const float sd = h8 ? a0 : a1;
    k += __shfl_xor_sync(0xffffffffu, sd, 8);
    k += __shfl_xor_sync(0xffffffffu, k, 4);
    k += __shfl_xor_sync(0xffffffffu, k, 2);
    k += __shfl_xor_sync(0xffffffffu, k, 1);
    return k;
}

// A warp's bounded wait for a stage: every lane polls the barrier (the wait
// orders the bulk-copied bytes before the lane's reads); false for the whole
// warp once any lane hit the deadline or the CTA aborted.
__device__ __forceinline__ bool sd_wait(uint64_t *bar, uint32_t parity, uint64_t deadline, volatile int *abort) {
    bool ok = true;
    while (!mbar_try(bar, parity)) {
        if (*abort || global_ns() > deadline) {
            ok = false;
            break;
        }
    }
    return __all_sync(0xffffffffu, ok);
}

template <class D, bool GROUPED, int NCMAX>
__global__ void __launch_bounds__((NCMAX + 1) * 32, 1) moe_decode_stream_kernel(const SdArgs a) {
    extern __shared__ uint8_t sraw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)sraw + 127) & ~(uintptr_t)127);
    uint8_t *ring = base;
    float *redA = reinterpret_cast<float *>(base + a.off_redA);   // [slot][pair][slab][gate|up]
    float *redB = reinterpret_cast<float *>(base + a.off_redB);   // [ai][row][slab]
    int4 *desc = reinterpret_cast<int4 *>(base + a.off_desc);     // [slot]
    int *slot_cnt = reinterpret_cast<int *>(base + a.off_desc + 16 * a.n_stages);   // [slot]
    uint64_t *full = reinterpret_cast<uint64_t *>(base + a.off_bar);
    uint64_t *empty = full + a.n_stages;
    __shared__ DecodeRouting rt;
    __shared__ volatile int abort_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NC = a.nc, NCT = NC * 32, NS = a.n_stages, SB = a.stage_bytes, NG = a.n_groups, GW = a.group_warps;
    constexpr int SPG = kSdSlotsPerGroup;
    const int n = a.K;   // S = 1: the token's K slots
    const uint64_t deadline = global_ns() + (uint64_t)a.timeout_ns;
    constexpr bool grouped = GROUPED;
    unsigned *exitc = a.ctr + 1, *arrived = a.ctr + 2;   // CTAs out, barrier arrivals

    // consumer lanes: their chunk of x (phase A) is loaded now and converted to
    // limbs after the routing below, so the producer starts copying first
    const int grp = warp / GW, gi = warp - grp * GW;
    const int slA = gi % a.nsA, subA = gi / a.nsA, GA = GW / a.nsA;
    const int cA = slA * 32 + lane;
    const bool okA = cA < a.cpr_gu;
    float xv[D::NIN];
    if (warp < NC)
        d4_load_chunk<D::NIN>(a.x, a.H, okA ? cA : (long long)a.cpr_gu + 1, xv, [](const auto *p) { return __ldg(p); });

    // ---- phase 0: distinct routed experts in ascending id order, weights summed
    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < NS; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], GW);
            slot_cnt[i] = 0;
            // the last 16 bytes of every slot stay zero: the scale that lanes
            // past the end of a row multiply by
            *reinterpret_cast<uint4 *>(ring + (size_t)(i + 1) * SB - 16) = make_uint4(0, 0, 0, 0);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    decode_route(rt, a.ids, a.w, n, a.n_experts, a.table, NC);
    if (rt.bad) {
        if (blockIdx.x == 0 && tid == 0) atomicCAS(a.err, 0, DEV_ERR_BAD_ID);
        return;
    }
    const int nact = rt.nact;
    const int rpcB = (a.H + gridDim.x - 1) / gridDim.x;
    const int oc0 = min(a.H, (int)blockIdx.x * rpcB), oc1 = min(a.H, oc0 + rpcB);
    // slot layouts: A = [gate codes RP rows][up codes RP rows][gate scales][up scales];
    // B = [codes: expert m of the group, row r][scales, same order]; scales only for grouped formats
    const int offA_u = a.RP * a.rs_gu, offA_sg = 2 * offA_u, offA_su = offA_sg + a.RP * a.ng_gu * 4;
    const int nsB = a.nsB, nsBW = (nsB + D::SPW - 1) / D::SPW;   // slab sets of SPW per down row

    if (warp == NC) {
        // ---------------- producer lanes: lane g feeds group g.  Phase-A stages are
        // dealt round robin over the groups of all CTAs; then the group's
        // phase-B stages (its experts g, g + NG, ..., RB rows each); then an end marker
        if (lane < NG) {
            const int g = lane;
            const int spe = (a.F + a.RP - 1) / a.RP;   // phase-A stages per routed expert
            const unsigned totalA = (unsigned)(nact * spe);
            const unsigned V = gridDim.x * (unsigned)NG;
            const int nstB = oc1 > oc0 ? (oc1 - oc0 + a.RB - 1) / a.RB : 0;
            const int ne = g < nact ? (nact - g + NG - 1) / NG : 0;   // experts of the group
            int i = 0;   // the group's stage counter
            unsigned idx = blockIdx.x * (unsigned)NG + g;
            int jB = 0;
            bool ok = true;
            while (ok) {
                const int s = g * SPG + i % SPG;
                if (i >= SPG && !mbar_wait(&empty[s], ((i / SPG) & 1) ^ 1, deadline, &abort_flag)) {
                    if (!abort_flag) {
                        abort_flag = 1;
                        atomicCAS(a.err, 0, DEV_ERR_TIMEOUT);
                    }
                    break;
                }
                uint8_t *dst = ring + (size_t)s * SB;
                if (idx < totalA) {
                    const int ai = (int)(idx / spe), j0 = (int)(idx - (unsigned)ai * spe) * a.RP;
                    const int w = min(a.RP, a.F - j0);
                    desc[s] = make_int4(SD_A, ai, j0, w);
                    const uint32_t cb = (uint32_t)(w * a.rs_gu);
                    const uint32_t sb = grouped ? (uint32_t)(w * a.ng_gu * 4) : 0u;
                    mbar_expect_tx(&full[s], 2 * cb + 2 * sb);
                    bulk_load(dst, rt.q[ai][0] + (size_t)j0 * a.rs_gu, cb, &full[s]);
                    bulk_load(dst + offA_u, rt.q[ai][1] + (size_t)j0 * a.rs_gu, cb, &full[s]);
                    if (sb) {
                        bulk_load(dst + offA_sg, rt.s[ai][0] + (size_t)j0 * a.ng_gu, sb, &full[s]);
                        bulk_load(dst + offA_su, rt.s[ai][1] + (size_t)j0 * a.ng_gu, sb, &full[s]);
                    }
                    idx += V;
                } else if (jB < nstB) {
                    const int r0 = oc0 + jB * a.RB, w = min(a.RB, oc1 - r0);
                    desc[s] = make_int4(SD_B, ne, r0, w);
                    const uint32_t cb = (uint32_t)(w * a.rs_d), sb = grouped ? (uint32_t)(w * a.ng_d * 4) : 0u;
                    if (ne > 0) {
                        mbar_expect_tx(&full[s], (uint32_t)ne * (cb + sb));
                        for (int m = 0; m < ne; m++) {
                            const int ai = g + m * NG;
                            bulk_load(dst + (size_t)m * cb, rt.q[ai][2] + (size_t)r0 * a.rs_d, cb, &full[s]);
                            if (sb)
                                bulk_load(dst + (size_t)ne * cb + (size_t)m * sb, rt.s[ai][2] + (size_t)r0 * a.ng_d, sb,
                                          &full[s]);
                        }
                    } else {
                        mbar_arrive(&full[s]);
                    }
                    jB++;
                } else {
                    desc[s] = make_int4(SD_END_B, 0, 0, 0);
                    mbar_arrive(&full[s]);   // end marker: no bytes
                    ok = false;
                }
                i++;
            }
            // every copy issued has landed before the CTA may exit
            const uint64_t dl2 = global_ns() + 200000000ull;
            volatile int no_abort = 0;
            for (int q = max(0, i - SPG); q < i; q++) mbar_wait(&full[g * SPG + q % SPG], (q / SPG) & 1, dl2, &no_abort);
        }
        return;
    }

    // ---------------- consumers: group grp's stages, in its own slots; a group
    // sees its phase-A stages first, then its phase-B stages, then its end marker
    const int nsA = a.nsA;
    const uint32_t ring_s = smem_addr(ring);
    const int zero_off = SB - 16;   // a zero float in every slot
    const int kk = lane >> 3;
    int i = 0;   // the group's stage counter
    bool live = true;
    {
        // phase A: this warp's pairs of a stage are subA + m GA; four rows per
        // iteration: gate p, up p, gate p + GA, up p + GA.  Offsets from the slot
        // base run with the iteration; lanes past the end of a row read row 0's
        // codes (their limbs are zero) and the slot's zero scale.
        D xd;
        const uint32_t mbA = d4_warp_maxbits<D::NIN>(xv);
        xd.set(xv, d4_exp(mbA));
        const float invA = d4_unscale(mbA, D::UNSCALE_EXTRA);   // back to units of x, after the reduction
        const int rs = a.rs_gu, ng4 = a.ng_gu * 4;
        const int q0 = okA ? subA * rs + cA * 16 : 0, q1 = okA ? GA * rs : 0, dq = okA ? 2 * GA * rs : 0;
        const int giA = okA ? (cA >> a.gshift_gu) : 0;
        const int s0 = okA ? offA_sg + subA * ng4 + giA * 4 : zero_off, s1 = okA ? GA * ng4 : 0;
        const int su = okA ? offA_su - offA_sg : 0, ds = okA ? 2 * GA * ng4 : 0;
        // partial sum of lane 8k: pair subA (k < 2) or subA + GA, gate (k even) or up
        const int r0 = ((subA + (kk < 2 ? 0 : GA)) * nsA + slA) * 2 + (kk & 1), dr = 2 * GA * nsA * 2;
        const int pk = subA + (kk < 2 ? 0 : GA);
        while (true) {
            const int s = grp * SPG + i % SPG;
            if (!sd_wait(&full[s], (uint32_t)((i / SPG) & 1), deadline, &abort_flag)) {
                if (lane == 0 && !abort_flag) {
                    abort_flag = 1;
                    atomicCAS(a.err, 0, DEV_ERR_TIMEOUT);
                }
                live = false;
                break;
            }
            const int4 d = desc[s];
            if (d.x != SD_A) break;   // stage i belongs to phase B (or is the end marker)
            const uint32_t sb = ring_s + (uint32_t)(s * SB);
            float *red = redA + s * a.RP * nsA * 2 + r0;
            uint32_t qa = sb + q0, sa = sb + s0;
            int pp = pk;
            // two iterations per trip (the second one dropped past the stage's
            // pairs), so the two reductions overlap with each other and with
            // the dot products
            for (int p0 = subA; p0 < d.w; p0 += 4 * GA) {
                const bool two = p0 + 2 * GA < d.w;
                const uint32_t qb = two ? qa + dq : qa, sb2 = two ? sa + ds : sa;
                const uint4 qq[4] = {lds128(qa), lds128(qa + offA_u), lds128(qa + q1), lds128(qa + q1 + offA_u)};
                const uint4 qr[4] = {lds128(qb), lds128(qb + offA_u), lds128(qb + q1), lds128(qb + q1 + offA_u)};
                float sc[4], sd[4];
                if constexpr (GROUPED) {
                    sc[0] = ldsf(sa);
                    sc[1] = ldsf(sa + su);
                    sc[2] = ldsf(sa + s1);
                    sc[3] = ldsf(sa + s1 + su);
                    sd[0] = ldsf(sb2);
                    sd[1] = ldsf(sb2 + su);
                    sd[2] = ldsf(sb2 + s1);
                    sd[3] = ldsf(sb2 + s1 + su);
                } else {
                    const float z = okA ? 1.f : 0.f;
                    const int ra = d.z + min(p0, d.w - 1), rb = d.z + min(p0 + GA, d.w - 1);
                    const int rc = d.z + min(p0 + 2 * GA, d.w - 1), rd = d.z + min(p0 + 3 * GA, d.w - 1);
                    sc[0] = __ldg(rt.s[d.y][0] + ra) * z;
                    sc[1] = __ldg(rt.s[d.y][1] + ra) * z;
                    sc[2] = __ldg(rt.s[d.y][0] + rb) * z;
                    sc[3] = __ldg(rt.s[d.y][1] + rb) * z;
                    sd[0] = __ldg(rt.s[d.y][0] + rc) * z;
                    sd[1] = __ldg(rt.s[d.y][1] + rc) * z;
                    sd[2] = __ldg(rt.s[d.y][0] + rd) * z;
                    sd[3] = __ldg(rt.s[d.y][1] + rd) * z;
                }
                float dd[4], de[4];
                xd.template dotn<4>(qq, dd);
                xd.template dotn<4>(qr, de);
                const float t = sd_warp_sum4(dd[0] * sc[0], dd[1] * sc[1], dd[2] * sc[2], dd[3] * sc[3], lane);
                const float t2 = sd_warp_sum4(de[0] * sd[0], de[1] * sd[1], de[2] * sd[2], de[3] * sd[3], lane);
                if ((lane & 7) == 0) {
                    if (pp < d.w) red[0] = t * invA;
                    if (pp + 2 * GA < d.w) red[dr] = t2 * invA;
                }
                qa += 2 * dq;
                sa += 2 * ds;
                red += 2 * dr;
                pp += 4 * GA;
            }
            // the last warp of the group to finish the stage turns its pairs into
            // h = silu(g) * u (plain stores; the grid barrier publishes them)
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                __threadfence_block();
                last = atomicAdd(&slot_cnt[s], 1) == GW - 1;
            }
            if (__shfl_sync(0xffffffffu, last, 0)) {
                __threadfence_block();
                const float *rd = redA + s * a.RP * nsA * 2;
                float *hrow = a.hbuf + (size_t)d.y * a.F + d.z;
                for (int q = lane; q < d.w; q += 32) {
                    float g = 0.f, u = 0.f;
                    for (int k2 = 0; k2 < nsA; k2++) {
                        g += rd[(q * nsA + k2) * 2];
                        u += rd[(q * nsA + k2) * 2 + 1];
                    }
                    hrow[q] = g / (1.0f + expf(-g)) * u;
                }
                if (lane == 0) slot_cnt[s] = 0;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            i++;
        }
    }
    // grid barrier among the consumers of all CTAs: every h is in global memory
    // after it (the producer keeps copying phase-B stages meanwhile)
    named_sync(1, NCT);
    if (tid == 0 && !abort_flag && !decode_grid_barrier(arrived, deadline, a.err)) abort_flag = 1;
    named_sync(1, NCT);
    // phase B: warp gi of group grp owns expert ai = grp + NG (gi / nsBW) and the
    // slabs SPW (gi % nsBW) ..; its h limbs are converted here, once
    if (live) {
        const int m = gi / nsBW, sw = gi - m * nsBW;
        const int ai = grp + NG * m;
        const bool active = ai < nact;
        D xb[D::SPW];
        float invB[D::SPW];
        bool okB[D::SPW];
        int qoffB[D::SPW], giB[D::SPW];
#pragma unroll
        for (int u = 0; u < D::SPW; u++) {
            const int slab = sw * D::SPW + u;
            const int cB = slab * 32 + lane;
            okB[u] = active && slab < nsB && cB < a.cpr_d;
            qoffB[u] = okB[u] ? cB * 16 : 0;
            giB[u] = okB[u] ? (cB >> a.gshift_d) : 0;
            float v[D::NIN];
            // L1-allocating loads: a lane reads all 128 bytes of one line, and the
            // grid barrier's acquire has dropped any older copy from this SM's L1
            d4_load_chunk<D::NIN>(a.hbuf + (size_t)(active ? ai : 0) * a.F, a.F, okB[u] ? cB : (long long)a.cpr_d + 1,
                                  v, [](const auto *p) { return __ldca(p); });
            const uint32_t mb = d4_warp_maxbits<D::NIN>(v);
            xb[u].set(v, d4_exp(mb));
            invB[u] = d4_unscale(mb, D::UNSCALE_EXTRA);
        }
        const int rsd = a.rs_d, ngd4 = a.ng_d * 4;
        while (true) {
            const int s = grp * SPG + i % SPG;
            if (!sd_wait(&full[s], (uint32_t)((i / SPG) & 1), deadline, &abort_flag)) {
                if (lane == 0 && !abort_flag) {
                    abort_flag = 1;
                    atomicCAS(a.err, 0, DEV_ERR_TIMEOUT);
                }
                break;
            }
            const int4 d = desc[s];
            if (d.x != SD_B) {   // end marker
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                break;
            }
            if (active && m < d.y) {
                const uint32_t sb = ring_s + (uint32_t)(s * SB);
                const int nr = d.w;
                const uint32_t cbase = sb + (uint32_t)(m * nr * rsd);
                const uint32_t sbase = sb + (uint32_t)(d.y * nr * rsd + m * nr * ngd4);
                float *rb = redB + (ai * rpcB + (d.z - oc0) + kk) * nsB;
#pragma unroll
                for (int u = 0; u < D::SPW; u++) {
                    const int slab = sw * D::SPW + u;
                    if (slab >= nsB) break;
                    // lanes past the end of a row: row 0's codes, the zero scale
                    uint32_t qa = cbase + qoffB[u];
                    uint32_t sa = okB[u] ? sbase + giB[u] * 4 : sb + zero_off;
                    const int dq = okB[u] ? rsd : 0, dsc = okB[u] ? ngd4 : 0;
                    float *rr = rb + slab;
                    int r0 = 0;
                    // eight rows per trip: two independent dot products and reductions
                    for (; r0 + 8 <= nr; r0 += 8) {
                        const uint4 qq[4] = {lds128(qa), lds128(qa + dq), lds128(qa + 2 * dq), lds128(qa + 3 * dq)};
                        const uint4 qr[4] = {lds128(qa + 4 * dq), lds128(qa + 5 * dq), lds128(qa + 6 * dq),
                                             lds128(qa + 7 * dq)};
                        float sc[8];
                        if constexpr (GROUPED) {
#pragma unroll
                            for (int q = 0; q < 8; q++) sc[q] = ldsf(sa + q * dsc);
                        } else {
                            const float *ps = rt.s[ai][2] + d.z + r0;
                            const float z = okB[u] ? 1.f : 0.f;
#pragma unroll
                            for (int q = 0; q < 8; q++) sc[q] = __ldg(ps + q) * z;
                        }
                        float dd[4], de[4];
                        xb[u].template dotn<4>(qq, dd);
                        xb[u].template dotn<4>(qr, de);
                        const float t = sd_warp_sum4(dd[0] * sc[0], dd[1] * sc[1], dd[2] * sc[2], dd[3] * sc[3], lane);
                        const float t2 = sd_warp_sum4(de[0] * sc[4], de[1] * sc[5], de[2] * sc[6], de[3] * sc[7], lane);
                        if ((lane & 7) == 0) {
                            rr[0] = t * invB[u];
                            rr[4 * nsB] = t2 * invB[u];
                        }
                        qa += 8 * dq;
                        sa += 8 * dsc;
                        rr += 8 * nsB;
                    }
                    for (; r0 + 4 <= nr; r0 += 4) {
                        const uint4 qq[4] = {lds128(qa), lds128(qa + dq), lds128(qa + 2 * dq), lds128(qa + 3 * dq)};
                        float sc[4];
                        if constexpr (GROUPED) {
                            sc[0] = ldsf(sa);
                            sc[1] = ldsf(sa + dsc);
                            sc[2] = ldsf(sa + 2 * dsc);
                            sc[3] = ldsf(sa + 3 * dsc);
                        } else {
                            const float *ps = rt.s[ai][2] + d.z + r0;
                            const float z = okB[u] ? 1.f : 0.f;
                            sc[0] = __ldg(ps) * z;
                            sc[1] = __ldg(ps + 1) * z;
                            sc[2] = __ldg(ps + 2) * z;
                            sc[3] = __ldg(ps + 3) * z;
                        }
                        float dd[4];
                        xb[u].template dotn<4>(qq, dd);
                        const float t = sd_warp_sum4(dd[0] * sc[0], dd[1] * sc[1], dd[2] * sc[2], dd[3] * sc[3], lane);
                        if ((lane & 7) == 0) *rr = t * invB[u];
                        qa += 4 * dq;
                        sa += 4 * dsc;
                        rr += 4 * nsB;
                    }
                    const int rem = nr - r0;   // 0..3 rows left
                    if (rem > 0) {
                        float v4[4] = {0.f, 0.f, 0.f, 0.f};
                        float sc[3];
#pragma unroll
                        for (int q = 0; q < 3; q++) {
                            const int rq = min(q, rem - 1);
                            if constexpr (GROUPED) sc[q] = ldsf(sa + rq * dsc);
                            else sc[q] = okB[u] ? __ldg(rt.s[ai][2] + d.z + r0 + rq) : 0.f;
                        }
                        if (rem == 1) {
                            const uint4 q1[1] = {lds128(qa)};
                            float d1[1];
                            xb[u].template dotn<1>(q1, d1);
                            v4[0] = d1[0] * sc[0];
                        } else if (rem == 2) {
                            const uint4 q2[2] = {lds128(qa), lds128(qa + dq)};
                            float d2[2];
                            xb[u].template dotn<2>(q2, d2);
                            v4[0] = d2[0] * sc[0];
                            v4[1] = d2[1] * sc[1];
                        } else {
                            const uint4 q3[3] = {lds128(qa), lds128(qa + dq), lds128(qa + 2 * dq)};
                            float d3[3];
                            xb[u].template dotn<3>(q3, d3);
                            v4[0] = d3[0] * sc[0];
                            v4[1] = d3[1] * sc[1];
                            v4[2] = d3[2] * sc[2];
                        }
                        const float t = sd_warp_sum4(v4[0], v4[1], v4[2], v4[3], lane);
                        if ((lane & 7) == 0 && kk < rem) *rr = t * invB[u];
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            i++;
        }
    }
    named_sync(1, NCT);
    for (int rr = tid; rr < oc1 - oc0; rr += NCT) {
        float acc = 0.f;
        for (int ai = 0; ai < nact; ai++) {
            float dsum = 0.f;
            for (int q = 0; q < nsB; q++) dsum += redB[(ai * rpcB + rr) * nsB + q];
            acc = fmaf(rt.ew[ai], dsum, acc);
        }
        a.y[oc0 + rr] = acc;
    }
    // the last CTA out resets the barrier counter for the next call, also after
    // an aborted call
    if (tid == 0) decode_exit(exitc, arrived);
}

template <class D, bool GROUPED, int NCMAX>
cudaError_t sd_launch_t(const SdArgs &a, int grid, size_t smem, cudaStream_t st) {
    auto kern = moe_decode_stream_kernel<D, GROUPED, NCMAX>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((a.nc + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <class D, bool GROUPED, int NCMAX>
cudaError_t sd_occupancy_t(int nc, size_t smem, int *per_sm) {
    auto kern = moe_decode_stream_kernel<D, GROUPED, NCMAX>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, kern, (nc + 1) * 32, smem);
}

constexpr int kSdNcNib = 19;    // consumer warps at most, int4: 20 warps, at most 5 per scheduler, 96 registers
constexpr int kSdNcByte = 24;   // consumer warps at most, int8: 25 warps, 72 registers

int gcd_i(int p, int q) { return q == 0 ? p : gcd_i(q, p % q); }

}  // namespace

// Geometry of the streamed decode block for an expert table (fmt 1, 2 or 4,
// rows of rs_gu / rs_d bytes, ng scales per row when grouped) on a GPU with
// n_sm SMs and smem_max bytes of shared memory per block.  Returns false when
// the table does not fit this kernel (the caller takes another one).
bool sd_plan(int fmt, int H, int F, int K, int cpr_gu, int cpr_d, int rs_gu, int rs_d, int ng_gu, int ng_d,
             int n_sm, size_t smem_max, SdArgs *a, size_t *smem) {
    const bool nib = fmt == 2 || fmt == 4;
    if (!nib && fmt != 1) return false;
    const bool grouped = fmt == 4;
    if (grouped && (ng_gu % 4 != 0 || ng_d % 4 != 0)) return false;   // 16-byte scale copies
    const int nsA = (cpr_gu + 31) / 32, nsB = (cpr_d + 31) / 32;
    const int spw = nib ? D4Nib::SPW : D4Byte::SPW, nsBW = (nsB + spw - 1) / spw;
    // a group has at least one warp per slab of a gate/up row and per slab set
    // of a down row (L); up to three groups, each with two slots of its own
    const int L = nsA / gcd_i(nsA, nsBW) * nsBW;
    const int ncmax = nib ? kSdNcNib : kSdNcByte;
    if (L > ncmax) return false;
    const int NG = std::min(3, ncmax / L);
    const int GW = (ncmax / NG) / L * L;
    const int NS = kSdSlotsPerGroup * NG;
    const int GA = GW / nsA;
    // phase B: every routed expert of a group needs nsBW warps of it
    const int ne_max = (K + NG - 1) / NG;
    if (ne_max * nsBW > GW) return false;
    const int rpcB = (H + n_sm - 1) / n_sm;
    const size_t rowB = (size_t)rs_d + (grouped ? 4 * ng_d : 0), rowA = 2 * ((size_t)rs_gu + (grouped ? 4 * ng_gu : 0));
    // fixed shared memory: partial sums, descriptors, barriers, static arrays, alignment
    const size_t fixed_guess = 12 * 1024 + (size_t)K * rpcB * nsB * 4;
    const size_t budget = smem_max > fixed_guess ? smem_max - fixed_guess : 0;
    const size_t slot_max = budget / NS;
    if (slot_max < 16 + ne_max * rowB || slot_max < 16 + 2 * GA * rowA) return false;
    // phase B: RB rows of each of a group's experts; phase A: whole iterations
    // (2 GA pairs) of every warp
    // phase-B stages of equal size: the fewest that hold a CTA's rows of one expert
    const int RBmax = (int)std::min<size_t>((size_t)rpcB, (slot_max - 16) / (ne_max * rowB));
    if (RBmax < 1) return false;
    const int nstB = (rpcB + RBmax - 1) / RBmax, RB = (rpcB + nstB - 1) / nstB;
    const int RP = std::min((int)((slot_max - 16) / rowA) / (2 * GA) * (2 * GA), 64 * GA);
    if (RB < 1 || RP < 1) return false;
    const size_t stA = (size_t)RP * rowA, stB = (size_t)RB * ne_max * rowB;
    const size_t SB = (std::max(stA, stB) + 16 + 127) / 128 * 128;
    const size_t redA = (size_t)NS * RP * nsA * 2 * 4, redB = (size_t)K * rpcB * nsB * 4;
    const size_t off_redA = NS * SB, off_redB = (off_redA + redA + 15) / 16 * 16;
    const size_t off_desc = (off_redB + redB + 15) / 16 * 16;
    const size_t off_bar = (off_desc + (size_t)NS * 16 + (size_t)NS * 4 + 15) / 16 * 16;
    const size_t total = off_bar + 2 * NS * 8 + 128;   // + alignment slack of the base
    // static shared memory of the kernel: about 3.9 KB
    if (total + 4096 > smem_max || SB > (1u << 30)) return false;
    memset(a, 0, sizeof *a);
    a->K = K;
    a->H = H;
    a->F = F;
    a->nc = NG * GW;   // <= ncmax
    a->n_groups = NG;
    a->group_warps = GW;
    a->nsA = nsA;
    a->nsB = nsB;
    a->cpr_gu = cpr_gu;
    a->cpr_d = cpr_d;
    a->rs_gu = rs_gu;
    a->rs_d = rs_d;
    a->ng_gu = grouped ? ng_gu : 1;
    a->ng_d = grouped ? ng_d : 1;
    a->grouped = grouped;
    a->RP = RP;
    a->RB = RB;
    a->stage_bytes = (int)SB;
    a->n_stages = NS;
    a->off_redA = (int)off_redA;
    a->off_redB = (int)off_redB;
    a->off_desc = (int)off_desc;
    a->off_bar = (int)off_bar;
    a->fmt = fmt;
    *smem = total;
    return true;
}

// Scratch of one call: h [K][F] floats.
size_t sd_scratch_bytes(const SdArgs &a) { return (size_t)a.K * a.F * 4; }
// Counter words of one call (zero between calls): unused, CTAs out, barrier
// arrivals.
size_t sd_counter_words(const SdArgs &) { return 4; }

cudaError_t sd_occupancy(const SdArgs &a, size_t smem, int *per_sm) {
    if (a.fmt == 1) return sd_occupancy_t<D4Byte, false, kSdNcByte>(a.nc, smem, per_sm);
    if (a.grouped) return sd_occupancy_t<D4Nib, true, kSdNcNib>(a.nc, smem, per_sm);
    return sd_occupancy_t<D4Nib, false, kSdNcNib>(a.nc, smem, per_sm);
}

cudaError_t launch_stream_decode(const SdArgs &a, int grid, size_t smem, cudaStream_t st) {
    if (a.fmt == 1) return sd_launch_t<D4Byte, false, kSdNcByte>(a, grid, smem, st);
    if (a.grouped) return sd_launch_t<D4Nib, true, kSdNcNib>(a, grid, smem, st);
    return sd_launch_t<D4Nib, false, kSdNcNib>(a, grid, smem, st);
}

}  // namespace coli

// CPU replay of the correlation kernel's launch plan and index arithmetic for one geometry
// (forward and backward-data): every weight tap used once, paired-tap offsets, staged rows
// within the blocked copy, weight blocks within the packed buffer, TMEM columns of the paired
// epilogue within one accumulator, every store inside the output, every output position
// covered by exactly one tile.  A stride-2 backward-data pass is checked both as one launch
// per output phase and as the single launch that carries every phase (with the zero fills,
// every dx position is then written exactly once).  Host code only: the library source is
// included and the few device-facing helpers it calls are stubbed.
// Usage: corr2_plan_replay <14 or 16 geometry ints>; exits non-zero and prints FAIL lines
// on any violation.
#include "../../bwd_gconv_fwd_gb300/csrc/tc_conv.cu"
#include <cstdio>
#include <cstdlib>
namespace gconv {
long long wait_limit() { return 1000000000LL; }
int num_sms() { return 152; }
unsigned int *device_error_word() { return nullptr; }
int forced_path() { return 0; }
int wgrad_tma_enabled() { return 1; }
void *debug_trace(size_t *b) { *b = 0; return nullptr; }
bool encode_rows_tmap(CUtensorMap *, const void *, uint64_t, uint64_t, uint32_t, uint64_t) { return false; }
}
using namespace gconv;
static long errors = 0;
#define CHECK(cond, ...) do { if (!(cond)) { if (errors++ < 10) { printf("FAIL: " __VA_ARGS__); printf("\n"); } } } while (0)

// Checks one launch.  seen: uses of each (channel chunk, weight tap), accumulated by the
// caller; written: writes of each dx / y element of image 0, group 0, channel 0 (phase
// cases), or nullptr.
static void check_launch(const Geom &g, int bd, const Corr2Launch &C, std::vector<int> &seen, std::vector<int> *written)
{
    const Corr2Params &c = C.cp;
    const Pack2Params &k = C.pk;
    const bool phase = c.o_sh > 1 || c.o_sw > 1;
    CHECK(c.nph >= 1 && c.nph <= kMaxPlanes, "phase count %d", c.nph);
    CHECK(c.ph_tile0[0] == 0 && c.ph_tile0[c.nph] == c.n_tiles, "phase tile ranges");
    CHECK(k.nblk == c.nblk && c.nblk <= kMaxBlk, "block counts");
    const int plane = c.R * c.Wp;
    const int srcH = bd ? g.Ho : g.H, srcW = bd ? g.Wo : g.W;
    for (int ph = 0; ph < c.nph; ++ph) {
        CHECK(c.ph_tile0[ph + 1] - c.ph_tile0[ph] == c.N * c.G * c.n_vtile * c.n_ptile[ph], "phase %d tiles", ph);
        CHECK(c.Qh[ph] * c.Wp <= plane && c.Qw[ph] <= c.Wp, "phase %d grid past the plane", ph);
        CHECK(c.blk0[ph][0] >= 0 && c.blk0[ph][c.nchu] <= c.nblk, "phase %d block range", ph);
        if (ph > 0) CHECK(c.blk0[ph][0] == c.blk0[ph - 1][c.nchu], "phase %d blocks not after phase %d's", ph, ph - 1);
        const int rh = phase ? c.o_rh[ph] : 0, rw = phase ? c.o_rw[ph] : 0;
        for (int kc = 0; kc < c.nchu; ++kc) {
            CHECK(c.blk0[ph][kc + 1] > c.blk0[ph][kc], "phase %d chunk %d without blocks", ph, kc);
            for (int b = c.blk0[ph][kc]; b < c.blk0[ph][kc + 1]; ++b) {
                CHECK(k.jc[b] == kc % c.nchc, "block %d channel chunk", b);
                seen[(size_t)k.jc[b] * g.kH * g.kW + k.tk1[b]]++;
                if (k.tk2[b] >= 0) seen[(size_t)k.jc[b] * g.kH * g.kW + k.tk2[b]]++;
                CHECK(c.tap_off[b] + c.nmma <= c.stage_rows, "B rows");
                if (k.tk2[b] >= 0) continue;
                // what each output position reads through the blocked copy is the source
                // element the definition pairs with that output and tap (or both lie outside)
                const int kh = k.tk1[b] / g.kW, kw = k.tk1[b] % g.kW;
                for (int qh = 0; qh < c.Qh[ph]; ++qh)
                    for (int qw = 0; qw < c.Qw[ph]; ++qw) {
                        const int row = qh * c.Wp + qw + c.tap_off[b];
                        CHECK(row < plane, "staged row past the plane");
                        const int r = row / c.Wp, cc = row % c.Wp;
                        int sh, sw;
                        if (C.bu.nchc > 0) {
                            const int pl = kc / C.bu.nchc;
                            sh = r * C.bu.sh + C.bu.roff[pl];
                            sw = cc * C.bu.sw + C.bu.coff[pl];
                        } else {
                            sh = r + C.bu.r_off;
                            sw = cc + C.bu.c_off;
                        }
                        int eh, ew;
                        if (!bd) {
                            eh = g.s_h * qh + kh * g.d_h - g.pt;
                            ew = g.s_w * qw + kw * g.d_w - g.pl;
                        } else if (!phase) {
                            eh = qh + g.pt - kh * g.d_h;
                            ew = qw + g.pl - kw * g.d_w;
                        } else {
                            // dx (qh*s + rh, qw*s + rw) takes gradOutput ((ih + pt - kh*d)/s, ...)
                            const int th = qh * g.s_h + rh + g.pt - kh * g.d_h;
                            const int tw = qw * g.s_w + rw + g.pl - kw * g.d_w;
                            CHECK(th % g.s_h == 0 && tw % g.s_w == 0, "phase tap (%d,%d) not exact", kh, kw);
                            eh = th < 0 ? -1 : th / g.s_h;
                            ew = tw < 0 ? -1 : tw / g.s_w;
                        }
                        const bool in_e = eh >= 0 && eh < srcH && ew >= 0 && ew < srcW;
                        const bool in_s = sh >= 0 && sh < srcH && sw >= 0 && sw < srcW;
                        CHECK(in_e == in_s && (!in_e || (eh == sh && ew == sw)),
                              "phase %d chunk %d block %d tap (%d,%d) output (%d,%d): reads (%d,%d), definition (%d,%d)", ph,
                              kc, b, kh, kw, qh, qw, sh, sw, eh, ew);
                    }
            }
        }
    }
    // pair semantics: second tap offset = first + pair_delta (recomputed from the tap indices)
    for (int b = 0; b < c.nblk; ++b)
        if (k.tk2[b] >= 0) {
            auto off = [&](int t) { const int kh = t / g.kW, kw = t % g.kW;
                const int a = bd ? (g.kH - 1 - kh) * g.d_h : kh * g.d_h, bb = bd ? (g.kW - 1 - kw) * g.d_w : kw * g.d_w; return a * c.Wp + bb; };
            CHECK(off(k.tk1[b]) == c.tap_off[b] && off(k.tk2[b]) == c.tap_off[b] + c.pair_delta, "pair offsets");
            CHECK(c.Cv <= 64 && c.n_vtile == 1, "pair needs one 64-row half");
        }
    // shared memory: staging buffers, ring slots of spb blocks, the epilogue's transposes
    CHECK(c.spb == 1 || c.spb == 2, "blocks a slot %d", c.spb);
    CHECK(c.wstages >= 3 && c.wstages <= kC2MaxWStages && (c.nsb == 1 || c.nsb == 2), "ring %d, buffers %d", c.wstages, c.nsb);
    CHECK(1024 + (size_t)c.nsb * c.stage_rows * 128 + (size_t)c.wstages * c.spb * kWblkBytes + kC2EpiBytes <= C.smem &&
              C.smem <= (size_t)kC2MaxSmem, "shared memory layout");
    // ring slots: the producers' order (chunk by chunk, spb consecutive blocks a slot) and the
    // issuer's (full slots, then a one-block slot where a chunk's count is odd) name the
    // same blocks, so every wait meets the copy it waits for
    for (int ph = 0; ph < c.nph; ++ph) {
        std::vector<std::pair<int, int>> prod, iss;   // (first block, blocks)
        for (int kc = 0; kc < c.nchu; ++kc) {
            const int b0 = c.blk0[ph][kc], jend = c.blk0[ph][kc + 1];
            CHECK(jend > b0, "phase %d chunk %d without blocks", ph, kc);
            for (int j = b0; j < jend; j += c.spb) prod.push_back({j, std::min(c.spb, jend - j)});
            const int nbk = jend - b0, nfull = nbk / c.spb;
            for (int i = 0; i < nfull; ++i) iss.push_back({b0 + i * c.spb, c.spb});
            if (nfull * c.spb < nbk) iss.push_back({b0 + nfull * c.spb, 1});
        }
        CHECK(prod == iss, "phase %d: producer and issuer slot sequences differ", ph);
    }
    // TMEM columns read by the epilogue stay in the 256-column buffer
    if (c.pair_delta) {
        int maxcol = 0;
        for (int pc = 0; pc < c.tile_pos; pc += 16) maxcol = std::max(maxcol, pc + c.pair_delta + 15);
        CHECK(maxcol <= 255, "upper TMEM column %d", maxcol);
    }
    const size_t out_elems = (size_t)c.N * c.G * c.Cv * c.oH * c.oW;
    const int64_t out_hw = (int64_t)c.oH * c.oW;
    std::vector<int> cov;
    for (int t = 0; t < c.n_tiles; ++t) {
        // the kernel's tile decode
        int ph = 0;
        while (ph + 1 < c.nph && t >= c.ph_tile0[ph + 1]) ++ph;
        int tt = t - c.ph_tile0[ph];
        const int ptile = tt % c.n_ptile[ph]; tt /= c.n_ptile[ph];
        const int n = tt % c.N; tt /= c.N;
        const int vt = tt % c.n_vtile;
        const int gg = tt / c.n_vtile;
        CHECK(gg < c.G, "tile %d group", t);
        const int p0 = ptile * c.tile_pos;
        for (int kc = 0; kc < c.nchu; ++kc)
            for (int m = 0; m < c.stage_rows; ++m)
                if (p0 + m < plane) {
                    const int64_t e = ((((int64_t)n * c.G + gg) * c.nchu + kc) * plane + p0 + m) * 64;
                    CHECK((size_t)(e + 64) * 2 <= C.ub_bytes, "stage src");
                }
        // the weight producers read blocks [blk0[ph][0], blk0[ph][nchu]) of (gg, vt)
        CHECK((((size_t)gg * c.n_vtile + vt) * c.nblk + c.blk0[ph][c.nchu]) * kWblkBytes <= C.wpk_bytes, "weights");
        // stores: each tile writes positions [p0, p0 + tile_pos) that are real outputs
        for (int j = 0; j < c.tile_pos; ++j) {
            const int pos = p0 + j, qh = pos / c.Wp, qw = pos % c.Wp;
            if (!(qh < c.Qh[ph] && qw < c.Qw[ph])) continue;
            const int oh = qh * c.o_sh + c.o_rh[ph], ow = qw * c.o_sw + c.o_rw[ph];
            CHECK(oh < c.oH && ow < c.oW, "store past the output plane");
            for (int vv = 0; vv < std::min(c.Cv, 128); ++vv) {
                const int64_t e = ((int64_t)n * c.G * c.Cv + (int64_t)gg * c.Cv + vt * 128 + vv) * out_hw + (int64_t)oh * c.oW + ow;
                CHECK(e >= 0 && (size_t)e < out_elems, "store");
            }
            if (written && n == 0 && gg == 0 && vt == 0) (*written)[(size_t)oh * c.oW + ow]++;
            if (!written && n == 0 && gg == 0 && vt == 0) {
                if (cov.empty()) cov.assign((size_t)c.oH * c.oW, 0);
                cov[(size_t)oh * c.oW + ow]++;
            }
        }
    }
    if (!written)
        for (size_t e = 0; e < cov.size(); ++e) CHECK(cov[e] == 1, "output %zu written %d times", e, cov[e]);
}

int main(int argc, char **argv)
{
    // 14 geometry integers (one stride, one dilation) or 16 (per axis)
    int v[16];
    if (argc == 15) {
        int a[14];
        for (int i = 0; i < 14; ++i) a[i] = atoi(argv[1 + i]);
        const int e[16] = {a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7], a[7], a[8], a[9], a[10], a[11], a[12], a[12], a[13]};
        for (int i = 0; i < 16; ++i) v[i] = e[i];
    } else {
        for (int i = 0; i < 16; ++i) v[i] = atoi(argv[1 + i]);
    }
    const int span_h = v[2] + v[9] + v[10] - v[13] * (v[5] - 1) - 1, span_w = v[3] + v[11] + v[12] - v[14] * (v[6] - 1) - 1;
    Geom g{v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7], v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15],
           span_h / v[7] + 1, span_w / v[8] + 1, v[1] / v[15], v[4] / v[15]};
    const bool strided = g.s_h != 1 || g.s_w != 1;
    // forward; stride-1 backward-data
    for (int bd = 0; bd < (strided ? 1 : 2); ++bd) {
        Corr2Launch C;
        if (!build_corr2(g, bd == 1, &C)) {
            printf("corr2 %d not served\n", bd);
            continue;
        }
        const Corr2Params &c = C.cp;
        printf("corr2 bwd_data=%d: Cv=%d pair_delta=%d nmma=%d tile_pos=%d blocks=%d stage_rows=%d tiles=%d smem=%zu\n",
               bd, c.Cv, c.pair_delta, c.nmma, c.tile_pos, c.nblk, c.stage_rows, c.n_tiles, C.smem);
        const int nchc = bd ? (g.Cgo + 63) / 64 : (g.Cgi + 63) / 64;
        std::vector<int> seen((size_t)g.kH * g.kW * nchc, 0);
        check_launch(g, bd, C, seen, nullptr);
        // every tap of every channel chunk once per stride plane it lies in (forward: each
        // tap lies in exactly one plane, so once in all)
        for (size_t t = 0; t < seen.size(); ++t) CHECK(seen[t] == 1, "tap %zu used %d times", t, seen[t]);
    }
    if (strided) {
        // stride-2 backward-data: the phase set, each phase alone and all phases in one launch
        Corr2PhaseSet S;
        if (!build_corr2_phases(g, &S)) {
            printf("corr2 phases not served\n");
        } else {
            const int nchc = (g.Cgo + 63) / 64;
            const size_t dx_plane = (size_t)g.H * g.W;
            for (int form = 0; form < 2; ++form) {
                if (form == 1 && !S.merged) break;
                std::vector<int> seen((size_t)g.kH * g.kW * nchc, 0);
                std::vector<int> written(dx_plane, 0);
                if (form == 0) {
                    for (int i = 0; i < S.n; ++i) {
                        CHECK(S.L[i].cp.nph == 1, "single-phase launch");
                        check_launch(g, 1, S.L[i], seen, &written);
                    }
                } else {
                    const Corr2Params &c = S.M.cp;
                    printf("merged phases: %d, blocks=%d nmma=%d stage_rows=%d tiles=%d smem=%zu ws=%zu\n", c.nph, c.nblk,
                           c.nmma, c.stage_rows, c.n_tiles, S.M.smem, S.ws_bytes);
                    CHECK(c.nph == S.n, "merged phase count");
                    CHECK(S.M.ws_bytes <= S.ws_bytes, "merged workspace");
                    check_launch(g, 1, S.M, seen, &written);
                }
                // zero fills: the dx positions of phases no tap reaches
                for (int z = 0; z < S.nzero; ++z)
                    for (int ih = S.zr[z]; ih < g.H; ih += g.s_h)
                        for (int iw = S.zc[z]; iw < g.W; iw += g.s_w) written[(size_t)ih * g.W + iw]++;
                for (size_t t = 0; t < seen.size(); ++t) CHECK(seen[t] == 1, "form %d: tap %zu used %d times", form, t, seen[t]);
                for (size_t e = 0; e < dx_plane; ++e) CHECK(written[e] == 1, "form %d: dx %zu written %d times", form, e, written[e]);
            }
            printf("phases: %d with taps, %d zero, merged=%d\n", S.n, S.nzero, (int)S.merged);
        }
    }
    printf("errors: %ld\n", errors);
    return errors ? 1 : 0;
}

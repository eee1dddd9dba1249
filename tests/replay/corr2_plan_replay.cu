// CPU replay of the correlation kernel's launch plan and index arithmetic for one geometry
// (forward and backward-data): every weight tap used once, paired-tap offsets, staged rows
// within the blocked copy, weight blocks within the packed buffer, TMEM columns of the paired
// epilogue within one accumulator, every store inside the output, every output position
// covered by exactly one tile.  Host code only: the library source is included and the few
// device-facing helpers it calls are stubbed.  Usage: corr2_plan_replay <14 geometry ints>;
// exits non-zero and prints FAIL lines on any violation.
#include "../../bwd_gconv_fwd_gb300/csrc/tc_conv.cu"
#include <cstdio>
#include <cstdlib>
namespace gconv {
long long wait_limit() { return 1000000000LL; }
int num_sms() { return 152; }
unsigned int *device_error_word() { return nullptr; }
int forced_path() { return 0; }
void *debug_trace(size_t *b) { *b = 0; return nullptr; }
bool encode_rows_tmap(CUtensorMap *, const void *, uint64_t, uint64_t, uint32_t, uint64_t) { return false; }
}
using namespace gconv;
static long errors = 0;
#define CHECK(cond, ...) do { if (!(cond)) { if (errors++ < 10) { printf("FAIL: " __VA_ARGS__); printf("\n"); } } } while (0)
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
    // the passes the correlation kernel serves: forward, stride-1 backward-data, and the
    // output phases of a stride-2 backward-data (each tap in exactly one phase)
    struct Case { int bd, rh, rw; };
    std::vector<Case> cases = {{0, -1, -1}};
    const bool strided = g.s_h != 1 || g.s_w != 1;
    if (!strided) cases.push_back({1, -1, -1});
    else
        for (int rh = 0; rh < g.s_h; ++rh)
            for (int rw = 0; rw < g.s_w; ++rw) cases.push_back({1, rh, rw});
    std::vector<int> seen_phases((size_t)g.kH * g.kW * 64, 0);
    bool any_phase = false;
    for (const Case &cs : cases) {
        const int bd = cs.bd;
        Corr2Launch C;
        bool no_taps = false;
        if (!build_corr2(g, bd == 1, &C, cs.rh, cs.rw, &no_taps)) {
            printf("corr2 %d (phase %d,%d) not served%s\n", bd, cs.rh, cs.rw, no_taps ? " (no taps)" : "");
            continue;
        }
        const bool phase = cs.rh >= 0;
        any_phase = any_phase || phase;
        const Corr2Params &c = C.cp;
        const Pack2Params &k = C.pk;
        printf("corr2 bwd_data=%d phase (%d,%d): Cv=%d pair_delta=%d nmma=%d tile_pos=%d blocks=%d stage_rows=%d tiles=%d smem=%zu\n",
               bd, cs.rh, cs.rw, c.Cv, c.pair_delta, c.nmma, c.tile_pos, c.nblk, c.stage_rows, c.n_tiles, C.smem);
        // every weight tap used exactly once for each 64-channel chunk of the reduced channels
        // (for the phases of a stride-2 backward-data: over all phases together)
        std::vector<int> seen_own((size_t)g.kH * g.kW * c.nchc, 0);
        std::vector<int> &seen = phase ? seen_phases : seen_own;
        CHECK(c.blk0[0] == 0 && c.blk0[c.nchu] == c.nblk && c.nblk <= kMaxBlk, "block ranges");
        for (int kc = 0; kc < c.nchu; ++kc) {
            CHECK(c.blk0[kc + 1] > c.blk0[kc], "chunk %d without blocks", kc);
            for (int b = c.blk0[kc]; b < c.blk0[kc + 1]; ++b) {
                CHECK(k.jc[b] == kc % c.nchc, "block %d channel chunk", b);
                seen[(size_t)k.jc[b] * g.kH * g.kW + k.tk1[b]]++;
                if (k.tk2[b] >= 0) seen[(size_t)k.jc[b] * g.kH * g.kW + k.tk2[b]]++;
                CHECK(c.tap_off[b] + c.nmma <= c.stage_rows, "B rows");
            }
        }
        if (!phase)
            for (size_t t = 0; t < seen.size(); ++t) CHECK(seen[t] == 1, "tap %zu used %d times", t, seen[t]);
        // what each (output position, unpaired block) reads, through the blocked copy, is the
        // source element the definition pairs with that output and tap (or both lie outside)
        const Geom &G0 = g;
        const int srcH = bd ? G0.Ho : G0.H, srcW = bd ? G0.Wo : G0.W;
        for (int kc = 0; kc < c.nchu; ++kc)
            for (int b = c.blk0[kc]; b < c.blk0[kc + 1]; ++b) {
                if (k.tk2[b] >= 0) continue;
                const int kh = k.tk1[b] / G0.kW, kw = k.tk1[b] % G0.kW;
                for (int qh = 0; qh < c.Qh; ++qh)
                    for (int qw = 0; qw < c.Qw; ++qw) {
                        const int row = qh * c.Wp + qw + c.tap_off[b];
                        CHECK(row < c.R * c.Wp, "staged row past the plane");
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
                            eh = G0.s_h * qh + kh * G0.d_h - G0.pt;
                            ew = G0.s_w * qw + kw * G0.d_w - G0.pl;
                        } else if (!phase) {
                            eh = qh + G0.pt - kh * G0.d_h;
                            ew = qw + G0.pl - kw * G0.d_w;
                        } else {
                            // dx (qh*s + rh, qw*s + rw) takes gradOutput ((ih + pt - kh*d)/s, ...)
                            const int th = qh * G0.s_h + cs.rh + G0.pt - kh * G0.d_h;
                            const int tw = qw * G0.s_w + cs.rw + G0.pl - kw * G0.d_w;
                            CHECK(th % G0.s_h == 0 && tw % G0.s_w == 0, "phase tap (%d,%d) not exact", kh, kw);
                            eh = th / G0.s_h;
                            ew = tw / G0.s_w;
                            if (th < 0) eh = -1;
                            if (tw < 0) ew = -1;
                        }
                        const bool in_e = eh >= 0 && eh < srcH && ew >= 0 && ew < srcW;
                        const bool in_s = sh >= 0 && sh < srcH && sw >= 0 && sw < srcW;
                        CHECK(in_e == in_s && (!in_e || (eh == sh && ew == sw)),
                              "chunk %d block %d tap (%d,%d) output (%d,%d): reads (%d,%d), definition (%d,%d)", kc, b, kh, kw,
                              qh, qw, sh, sw, eh, ew);
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
        // TMEM columns read by the epilogue stay in the 256-column buffer
        if (c.pair_delta) {
            int maxcol = 0;
            for (int pc = 0; pc < c.tile_pos; pc += 16) maxcol = std::max(maxcol, pc + c.pair_delta + 15);
            CHECK(maxcol <= 255, "upper TMEM column %d", maxcol);
        }
        const int plane = c.R * c.Wp;
        const size_t out_elems = (size_t)c.N * c.G * c.Cv * c.oH * c.oW;
        const int64_t out_hw = (int64_t)c.oH * c.oW;
        for (int t = 0; t < c.n_tiles; ++t) {
            int tt = t;
            const int ptile = tt % c.n_ptile; tt /= c.n_ptile;
            const int n = tt % c.N; tt /= c.N;
            const int vt = tt % c.n_vtile;
            const int gg = tt / c.n_vtile;
            const int p0 = ptile * c.tile_pos;
            for (int kc = 0; kc < c.nchu; ++kc)
                for (int m = 0; m < c.stage_rows; ++m)
                    if (p0 + m < plane) {
                        const int64_t e = ((((int64_t)n * c.G + gg) * c.nchu + kc) * plane + p0 + m) * 64;
                        CHECK((size_t)(e + 64) * 2 <= C.ub_bytes, "stage src");
                    }
            CHECK((((size_t)gg * c.n_vtile + vt) + 1) * c.nblk * kWblkBytes <= C.wpk_bytes, "weights");
            // stores: each tile writes positions [p0, p0 + tile_pos) that are real outputs
            const int cols = c.tile_pos;
            for (int j = 0; j < cols; ++j) {
                const int pos = p0 + j, qh = pos / c.Wp, qw = pos % c.Wp;
                if (!(qh < c.Qh && qw < c.Qw)) continue;
                for (int vv = 0; vv < std::min(c.Cv, 128); ++vv) {
                    const int oh = qh * c.o_sh + c.o_rh, ow = qw * c.o_sw + c.o_rw;
                    CHECK(oh < c.oH && ow < c.oW, "store past the output plane");
                    const int64_t e = ((int64_t)n * c.G * c.Cv + (int64_t)gg * c.Cv + vt * 128 + vv) * out_hw + (int64_t)oh * c.oW + ow;
                    CHECK(e >= 0 && (size_t)e < out_elems, "store");
                }
            }
        }
        // coverage: every real output position belongs to exactly one tile
        std::vector<int> cov(plane, 0);
        for (int pt = 0; pt < c.n_ptile; ++pt)
            for (int j = 0; j < c.tile_pos; ++j) if (pt * c.tile_pos + j < plane) cov[pt * c.tile_pos + j]++;
        for (int pos = 0; pos < c.Qh * c.Wp; ++pos) if (pos % c.Wp < c.Qw) CHECK(cov[pos] == 1, "coverage %d: %d", pos, cov[pos]);
    }
    if (any_phase) {
        // each tap of each channel chunk in exactly one stride-2 backward-data phase
        const int nchc = ((g.Cgo) + 63) / 64;
        for (size_t t = 0; t < (size_t)g.kH * g.kW * nchc; ++t) CHECK(seen_phases[t] == 1, "phase tap %zu used %d times", t, seen_phases[t]);
    }
    printf("errors: %ld\n", errors);
    return errors ? 1 : 0;
}

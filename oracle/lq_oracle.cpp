// lq_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, fp64 CPU statement of what the block-quantized decode matvec
// computes.  It exists so that the CUDA library can be checked against
// something written independently of it: it shares no source, header, table or
// helper with the library, and the library never calls it.  Only the tests,
// the smoke check and the bench's CPU-baseline leg load it.
//
// Sources (the pages this follows):
//  * larql "Architecture -> Metal shader map": the per-architecture tables
//    name the quantized matvecs (q4k_matvec, q6k_matvec, q4k_q6k_qkv_proj,
//    q4k_ffn_gate_up + geglu) and the dispatch-predicate table fixes the Q4_K
//    block at 144 bytes ("Q4_KF ... 144-byte block layout").
//  * dotLLM PR #320: the Q8_0 GEMV row-stride fix commit fixes a Q8_0 block at
//    34 bytes per 32 weights (row stride = blocksPerRow * 34); the LoRA Q8_0
//    commit gives the 32-element group; the MoE commit (MoeSwiGluMlp) fixes
//    the routing rule: softmax over all experts, top-k with the lower index
//    winning ties, renormalise by the sum of the selected probabilities, then
//    the weighted sum of per-expert SwiGLU FFNs.
//  * dotLLM PR #320, Qwen-MoE commit: norm_topk_prob = false keeps the
//    selected experts' softmax probabilities as weights (no renormalisation),
//    and an optional shared-expert SwiGLU branch is added to the routed sum,
//    scaled by sigmoid(x . shared_expert_gate) when that gate exists; the
//    follow-up commit allows N shared experts, summed.  Read here: the gate
//    scales the sum of the shared experts (one expert: the same either way).
//  * larql "Architecture -> Metal shader map", Gemma 3 table, row "Input
//    RMS-norm": a standard RMS-norm whose weight already carries the offset
//    (HF convention), the step the opt-in NORMED QKV variant fuses in front
//    of the projection: x_i * w_i / sqrt(mean_j x_j^2 + eps).
//  * dotLLM PR #255 (attention soft-cap: a score s becomes softCap *
//    tanh(s / softCap)) and PR #274 (FinalLogitSoftcap: the same map applied
//    to the logits after the lm_head GEMM): the final-logit soft-cap.
//  * The byte layout inside a Q4_K / Q6_K super-block is not printed on the
//    pages; this file takes the GGUF convention (the "GGUF-direct extract" of
//    the larql dispatch table).  Parity with real GGUF bytes is therefore
//    unpinned: no GGUF file is available to compare with.
//
// Everything here is written for obviousness, not speed: one weight at a time,
// in index order, in double precision.  Compiled with -ffp-contract=off so the
// x86 and Arm builds give the same doubles.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

const int FMT_Q4_K = 1;
const int FMT_Q6_K = 2;
const int FMT_Q8_0 = 3;

// IEEE-754 binary16 -> double, from the definition of the format:
// 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0) {
        v = std::ldexp((double)f, -24);               // subnormal: f * 2^-10 * 2^-14
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = std::ldexp((double)(1024 + f), e - 25);   // (1 + f/1024) * 2^(e-15)
    }
    return sign ? -v : v;
}

uint16_t read_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

// ---- Q4_K: 144 bytes = d (fp16) | dmin (fp16) | scales[12] | qs[128] -------
// Sub-block j (32 weights) has a 6-bit scale sc_j and a 6-bit min m_j packed
// in scales[12]: j < 4 -> low 6 bits of bytes j and j+4; j >= 4 -> low nibble
// / high nibble of byte j+4 for the four low bits, and the top two bits of
// bytes j-4 / j for the two high bits.
void q4k_scale_min(const uint8_t* s, int j, int* sc, int* m) {
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

// weight i of the super-block: quants come in four 32-byte groups; byte
// qs[32g + l] holds weight 64g + l in its low nibble and 64g + 32 + l in its
// high nibble.  w = d*sc*q - dmin*m, each product exact, one fp32 rounding.
void q4k_dequant_block(const uint8_t* blk, float* out) {
    double d = half_to_double(read_u16(blk));
    double dmin = half_to_double(read_u16(blk + 2));
    const uint8_t* s = blk + 4;
    const uint8_t* qs = blk + 16;
    for (int i = 0; i < 256; ++i) {
        int g = i / 64, within = i % 64;
        int q, j;
        if (within < 32) {
            q = qs[32 * g + within] & 15;
            j = 2 * g;
        } else {
            q = qs[32 * g + within - 32] >> 4;
            j = 2 * g + 1;
        }
        int sc, m;
        q4k_scale_min(s, j, &sc, &m);
        out[i] = (float)(d * sc * q - dmin * m);
    }
}

// ---- Q6_K: 210 bytes = ql[128] | qh[64] | int8 scales[16] | d (fp16) -------
// Two halves of 128 weights; half h uses ql[64h..], qh[32h..].  For l < 32:
//   weight 128h+l    = low nibble of ql[64h+l]    | bits 0-1 of qh[32h+l] << 4
//   weight 128h+32+l = low nibble of ql[64h+32+l] | bits 2-3 of qh[32h+l] << 4
//   weight 128h+64+l = high nibble of ql[64h+l]   | bits 4-5 of qh[32h+l] << 4
//   weight 128h+96+l = high nibble of ql[64h+32+l]| bits 6-7 of qh[32h+l] << 4
// each minus 32; weight i uses scale[i/16].  w = d*scale*q (exact in fp32).
void q6k_dequant_block(const uint8_t* blk, float* out) {
    const uint8_t* ql = blk;
    const uint8_t* qh = blk + 128;
    const int8_t* sc = (const int8_t*)(blk + 192);
    double d = half_to_double(read_u16(blk + 208));
    for (int i = 0; i < 256; ++i) {
        int h = i / 128, r = i % 128, quarter = r / 32, l = r % 32;
        int lowbyte = ql[64 * h + (quarter & 1) * 32 + l];
        int nib = (quarter < 2) ? (lowbyte & 15) : (lowbyte >> 4);
        int hi2 = (qh[32 * h + l] >> (2 * quarter)) & 3;
        int q = (nib | (hi2 << 4)) - 32;
        out[i] = (float)(d * sc[i / 16] * q);
    }
}

// ---- Q8_0: 34 bytes = d (fp16) | int8 qs[32];  w = d*q ----------------------
void q80_dequant_block(const uint8_t* blk, float* out) {
    double d = half_to_double(read_u16(blk));
    const int8_t* qs = (const int8_t*)(blk + 2);
    for (int i = 0; i < 32; ++i) out[i] = (float)(d * qs[i]);
}

int block_bytes(int fmt) {
    return fmt == FMT_Q4_K ? 144 : fmt == FMT_Q6_K ? 210 : fmt == FMT_Q8_0 ? 34 : 0;
}
int block_elems(int fmt) {
    return fmt == FMT_Q4_K ? 256 : fmt == FMT_Q6_K ? 256 : fmt == FMT_Q8_0 ? 32 : 0;
}

void dequant_row(int fmt, const uint8_t* row, int64_t cols, float* out) {
    int64_t nb = cols / block_elems(fmt);
    int bb = block_bytes(fmt), be = block_elems(fmt);
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t* blk = row + b * bb;
        float* o = out + b * be;
        if (fmt == FMT_Q4_K) q4k_dequant_block(blk, o);
        else if (fmt == FMT_Q6_K) q6k_dequant_block(blk, o);
        else q80_dequant_block(blk, o);
    }
}

double gelu_tanh(double g) {
    const double k = std::sqrt(2.0 / M_PI);
    return 0.5 * g * (1.0 + std::tanh(k * (g + 0.044715 * g * g * g)));
}
double silu(double g) { return g / (1.0 + std::exp(-g)); }

// Run fn(r0, r1) over [0, rows) split across nthreads std::threads.
template <class F>
void parallel_rows(int64_t rows, int nthreads, F fn) {
    if (nthreads <= 1 || rows < 2) {
        fn((int64_t)0, rows);
        return;
    }
    std::vector<std::thread> th;
    int64_t per = (rows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        int64_t r0 = t * per, r1 = std::min(rows, r0 + per);
        if (r0 >= r1) break;
        th.emplace_back([=] { fn(r0, r1); });
    }
    for (auto& t : th) t.join();
}

// y[b][r] = sum_j w_rj x[b][j] (index order, fp64); S = sum_j |w_rj x[b][j]|.
void matvec_row(int fmt, const uint8_t* W, int64_t cols, int64_t r, const float* x,
                int batch, double* y, double* S, int64_t rows_out, int64_t out_r,
                std::vector<float>& wrow) {
    int64_t rb = cols / block_elems(fmt) * block_bytes(fmt);
    dequant_row(fmt, W + r * rb, cols, wrow.data());
    for (int b = 0; b < batch; ++b) {
        const float* xb = x + (int64_t)b * cols;
        double acc = 0.0, sabs = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double t = (double)wrow[j] * (double)xb[j];
            acc += t;
            sabs += std::fabs(t);
        }
        y[(int64_t)b * rows_out + out_r] = acc;
        if (S) S[(int64_t)b * rows_out + out_r] = sabs;
    }
}

}  // namespace

extern "C" {

int orc_block_bytes(int fmt) { return block_bytes(fmt); }
int orc_block_elems(int fmt) { return block_elems(fmt); }
double orc_half_to_double(uint16_t h) { return half_to_double(h); }
double orc_gelu_tanh(double g) { return gelu_tanh(g); }
double orc_silu(double g) { return silu(g); }

// RMS-norm of ntok rows of n values: out = x * w / sqrt(mean(x^2) + eps).
void orc_rmsnorm(const float* X, int ntok, int64_t n, const float* w, double eps, double* out) {
    for (int t = 0; t < ntok; ++t) {
        const float* x = X + (int64_t)t * n;
        double ss = 0.0;
        for (int64_t j = 0; j < n; ++j) ss += (double)x[j] * (double)x[j];
        const double r = 1.0 / std::sqrt(ss / (double)n + eps);
        for (int64_t j = 0; j < n; ++j) out[(int64_t)t * n + j] = (double)x[j] * r * (double)w[j];
    }
}

// Final-logit soft-cap of n values: out[i] = cap * tanh(y[i] / cap).
void orc_softcap(const double* y, int64_t n, double cap, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = cap * std::tanh(y[i] / cap);
}

// Dequantize rows x cols weights (row-major block rows) to fp32.
void orc_dequant(int fmt, const uint8_t* W, int64_t rows, int64_t cols, float* out,
                 int nthreads) {
    int64_t rb = cols / block_elems(fmt) * block_bytes(fmt);
    parallel_rows(rows, nthreads, [&](int64_t r0, int64_t r1) {
        for (int64_t r = r0; r < r1; ++r) dequant_row(fmt, W + r * rb, cols, out + r * cols);
    });
}

// y = dequant(W) . x for a batch of x rows.  x: [batch][cols] fp32,
// y and S: [batch][rows] fp64.  S may be null.
void orc_matvec(int fmt, const uint8_t* W, int64_t rows, int64_t cols, const float* x,
                int batch, double* y, double* S, int nthreads) {
    parallel_rows(rows, nthreads, [&](int64_t r0, int64_t r1) {
        std::vector<float> wrow(cols);
        for (int64_t r = r0; r < r1; ++r)
            matvec_row(fmt, W, cols, r, x, batch, y, S, rows, r, wrow);
    });
}

// The same for a chosen list of rows only: y, S are [batch][nidx].
void orc_matvec_rows(int fmt, const uint8_t* W, int64_t cols, const int64_t* row_idx,
                     int64_t nidx, const float* x, int batch, double* y, double* S,
                     int nthreads) {
    parallel_rows(nidx, nthreads, [&](int64_t i0, int64_t i1) {
        std::vector<float> wrow(cols);
        for (int64_t i = i0; i < i1; ++i)
            matvec_row(fmt, W, cols, row_idx[i], x, batch, y, S, nidx, i, wrow);
    });
}

// Gated FFN front half: g = Wg.x, u = Wu.x, h = act(g) * u  (act applied to
// the gate; act = 1 -> GELU-tanh (GEGLU), 2 -> SiLU (SwiGLU)).  Outputs are
// [batch][inter] fp64; Sg, Su (may be null) the |w x| sums of g and u.
void orc_ffn_gate_up(int fmt, const uint8_t* Wg, const uint8_t* Wu, int64_t inter,
                     int64_t cols, const float* x, int batch, int act, double* h, double* g,
                     double* u, double* Sg, double* Su, int nthreads) {
    orc_matvec(fmt, Wg, inter, cols, x, batch, g, Sg, nthreads);
    orc_matvec(fmt, Wu, inter, cols, x, batch, u, Su, nthreads);
    for (int64_t i = 0; i < (int64_t)batch * inter; ++i) {
        double a = act == 1 ? gelu_tanh(g[i]) : silu(g[i]);
        h[i] = a * u[i];
    }
}

// MoE routing for ntok tokens: logits l_e = R_e . x (fp64), p = softmax(l),
// top-k by repeated maximum with the lower expert index winning ties,
// weights renormalised by the sum of the selected probabilities.
// idx, w: [ntok][topk]; logits, labs: [ntok][E] (labs = sum |R_ej x_j|).
void orc_moe_route(const float* R, int E, int64_t hidden, const float* X, int ntok, int topk,
                   int32_t* idx, double* w, double* logits, double* labs) {
    std::vector<double> l(E), p(E);
    std::vector<char> taken(E);
    for (int t = 0; t < ntok; ++t) {
        const float* x = X + (int64_t)t * hidden;
        for (int e = 0; e < E; ++e) {
            double acc = 0.0, sabs = 0.0;
            for (int64_t j = 0; j < hidden; ++j) {
                double v = (double)R[(int64_t)e * hidden + j] * (double)x[j];
                acc += v;
                sabs += std::fabs(v);
            }
            l[e] = acc;
            if (logits) logits[(int64_t)t * E + e] = acc;
            if (labs) labs[(int64_t)t * E + e] = sabs;
        }
        double mx = l[0];
        for (int e = 1; e < E; ++e) mx = std::max(mx, l[e]);
        double z = 0.0;
        for (int e = 0; e < E; ++e) {
            p[e] = std::exp(l[e] - mx);
            z += p[e];
        }
        for (int e = 0; e < E; ++e) p[e] /= z;
        for (int e = 0; e < E; ++e) taken[e] = 0;
        double sel = 0.0;
        for (int k = 0; k < topk; ++k) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || p[e] > p[best])) best = e;
            taken[best] = 1;
            idx[t * topk + k] = best;
            sel += p[best];
        }
        for (int k = 0; k < topk; ++k) w[t * topk + k] = p[idx[t * topk + k]] / sel;
    }
}

// Routing weights of a given selection: p = softmax(l) over all E experts,
// w_k = p_{idx_k} / sum of the selected p (renormalised by the sum).
void orc_moe_weights(const double* logits, int E, int ntok, const int32_t* idx, int topk,
                     double* w) {
    for (int t = 0; t < ntok; ++t) {
        const double* l = logits + (int64_t)t * E;
        double mx = l[0];
        for (int e = 1; e < E; ++e) mx = std::max(mx, l[e]);
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += std::exp(l[e] - mx);
        double sel = 0.0;
        for (int k = 0; k < topk; ++k) sel += std::exp(l[idx[t * topk + k]] - mx) / z;
        for (int k = 0; k < topk; ++k)
            w[t * topk + k] = (std::exp(l[idx[t * topk + k]] - mx) / z) / sel;
    }
}

// Routing weights without renormalisation (norm_topk_prob = false):
// w_k = p_{idx_k}, p = softmax(l) over all E experts.
void orc_moe_weights_raw(const double* logits, int E, int ntok, const int32_t* idx, int topk,
                         double* w) {
    for (int t = 0; t < ntok; ++t) {
        const double* l = logits + (int64_t)t * E;
        double mx = l[0];
        for (int e = 1; e < E; ++e) mx = std::max(mx, l[e]);
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += std::exp(l[e] - mx);
        for (int k = 0; k < topk; ++k) w[t * topk + k] = std::exp(l[idx[t * topk + k]] - mx) / z;
    }
}

// Shared-expert branch of an MoE layer: for token t,
//   S_t = gate_t * sum_s Wd_s (silu(Wg_s x_t) * (Wu_s x_t)),
//   gate_t = sigmoid(sum_j g_j x_tj) if g is given, else 1.
// nshared experts, each inter_s x hidden (Wg, Wu) and hidden x inter_s (Wd),
// all fmt.  S: [ntok][hidden], gscale: [ntok] (gate_t), fp64.
void orc_moe_shared(int fmt, const uint8_t* const* Wg, const uint8_t* const* Wu,
                    const uint8_t* const* Wd, int nshared, int64_t hidden, int64_t inter_s,
                    const float* X, int ntok, const float* g, double* S, double* gscale,
                    int nthreads) {
    std::vector<double> h(inter_s), gg(inter_s), uu(inter_s);
    std::vector<float> wrow(inter_s);
    const int64_t rb = inter_s / block_elems(fmt) * block_bytes(fmt);
    for (int t = 0; t < ntok; ++t) {
        const float* x = X + (int64_t)t * hidden;
        double gate = 1.0;
        if (g) {
            double z = 0.0;
            for (int64_t j = 0; j < hidden; ++j) z += (double)g[j] * (double)x[j];
            gate = 1.0 / (1.0 + std::exp(-z));
        }
        gscale[t] = gate;
        double* St = S + (int64_t)t * hidden;
        for (int64_t o = 0; o < hidden; ++o) St[o] = 0.0;
        for (int sh = 0; sh < nshared; ++sh) {
            orc_ffn_gate_up(fmt, Wg[sh], Wu[sh], inter_s, hidden, x, 1, 2, h.data(), gg.data(), uu.data(),
                            nullptr, nullptr, nthreads);
            for (int64_t o = 0; o < hidden; ++o) {
                dequant_row(fmt, Wd[sh] + o * rb, inter_s, wrow.data());
                double acc = 0.0;
                for (int64_t j = 0; j < inter_s; ++j) acc += (double)wrow[j] * h[j];
                St[o] += acc;
            }
        }
        for (int64_t o = 0; o < hidden; ++o) St[o] *= gate;
    }
}

// MoE expert FFN given a routing (idx, w): for token t,
//   Y_t = sum_k w_tk * W2_e (silu(W1_e x_t) * (W3_e x_t)),  e = idx[t][k]
// (w1 = gate, w3 = up, w2 = down, Mixtral naming).  Y: [ntok][hidden].
// Per routed slot s = t*topk + k the intermediate values are returned too:
// g, u, h, Sg, Su: [slot][inter];  ye, Sy: [slot][hidden] (expert output and
// its sum |w2_ij h_j|).  All fp64, all required.
void orc_moe_ffn(int fmt, const uint8_t* const* W1, const uint8_t* const* W3,
                 const uint8_t* const* W2, int64_t hidden, int64_t inter, const float* X,
                 int ntok, int topk, const int32_t* idx, const double* w, double* Y,
                 double* ye, double* Sy, double* hbuf, double* gbuf, double* ubuf,
                 double* Sg, double* Su, int nthreads) {
    std::vector<float> w2row(inter);
    for (int t = 0; t < ntok; ++t) {
        for (int64_t o = 0; o < hidden; ++o) Y[(int64_t)t * hidden + o] = 0.0;
        for (int k = 0; k < topk; ++k) {
            int e = idx[t * topk + k];
            int64_t slot = (int64_t)t * topk + k;
            double* h = hbuf + slot * inter;
            double* g = gbuf + slot * inter;
            double* u = ubuf + slot * inter;
            orc_ffn_gate_up(fmt, W1[e], W3[e], inter, hidden, X + (int64_t)t * hidden, 1, 2, h,
                            g, u, Sg ? Sg + slot * inter : nullptr,
                            Su ? Su + slot * inter : nullptr, nthreads);
            int64_t rb = inter / block_elems(fmt) * block_bytes(fmt);
            for (int64_t o = 0; o < hidden; ++o) {
                dequant_row(fmt, W2[e] + o * rb, inter, w2row.data());
                double acc = 0.0, sabs = 0.0;
                for (int64_t j = 0; j < inter; ++j) {
                    double v = (double)w2row[j] * h[j];
                    acc += v;
                    sabs += std::fabs(v);
                }
                if (ye) ye[slot * hidden + o] = acc;
                if (Sy) Sy[slot * hidden + o] = sabs;
                Y[(int64_t)t * hidden + o] += w[slot] * acc;
            }
        }
    }
}

// sum_j |w_ij| * v_j for every row i (rows x cols weights, v fp64 [cols]);
// used to carry a per-element bound on a matvec's input through the matvec.
void orc_abs_matvec(int fmt, const uint8_t* W, int64_t rows, int64_t cols, const double* v,
                    double* out, int nthreads) {
    int64_t rb = cols / block_elems(fmt) * block_bytes(fmt);
    parallel_rows(rows, nthreads, [&](int64_t r0, int64_t r1) {
        std::vector<float> wrow(cols);
        for (int64_t r = r0; r < r1; ++r) {
            dequant_row(fmt, W + r * rb, cols, wrow.data());
            double acc = 0.0;
            for (int64_t j = 0; j < cols; ++j) acc += std::fabs((double)wrow[j]) * v[j];
            out[r] = acc;
        }
    });
}

}  // extern "C"

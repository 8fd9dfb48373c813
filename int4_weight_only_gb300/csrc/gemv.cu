// gemv.cu - decode planner (plan_gemv) and the launches of the unsplit W4A16
// kernels and of the W4A8 kernels; the kernels are in gemv_impl.cuh.
#include "gemv_impl.cuh"

#include <array>

namespace w4 {

bool gemv_tma_activations(const GemvPlan& p) {
    const char* e = std::getenv("W4_GEMV_XTMA");
    if (e) return std::atoi(e) == 1;
    return !p.f16;
}

namespace {
bool plan_gemv_search(int M, int N, int Kp, int G, int act_bytes, int sm_count, GemvPlan* out,
                      int groups);
}

// Plans are cached by their inputs and the tuning variables' values, so
// repeated calls of one layer skip the search.
bool plan_gemv(int M, int N, int Kp, int G, int act_bytes, int sm_count, GemvPlan* out,
               int groups) {
    auto env = [](const char* n) {       // unset: 0; set: 1 + its value
        const char* e = std::getenv(n);
        return e ? 1 + std::atoi(e) : 0;
    };
    const std::array<int, 12> key = {M, N, Kp, G, act_bytes, sm_count, env("W4_GEMV_ROWS"),
                                     env("W4_GEMV_SPLIT"), env("W4_GEMV_CPS"),
                                     env("W4_GEMV_F16"), env("W4_GEMV_CSPLIT"), groups};
    static std::mutex mu;
    static std::map<std::array<int, 12>, std::pair<bool, GemvPlan>> cache;
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            if (it->second.first) *out = it->second.second;
            return it->second.first;
        }
    }
    GemvPlan p;
    const bool ok = plan_gemv_search(M, N, Kp, G, act_bytes, sm_count, &p, groups);
    std::lock_guard<std::mutex> lk(mu);
    if (cache.size() > 4096) cache.clear();
    cache[key] = {ok, p};
    if (ok) *out = p;
    return ok;
}

namespace {
bool plan_gemv_search(int M, int N, int Kp, int G, int act_bytes, int sm_count, GemvPlan* out,
                      int groups) {
    if (M < 1 || M > 16 || N < 1 || Kp < 1 || G < 32 || sm_count < 1) return false;
    const int pad = act_bytes == 2 ? 64 : 16;
    // W4A16 inner loop: fp16 for one or two tokens with groups of 64 or more
    // columns (its unpacking takes the fewest ALU operations per weight, and
    // its per-group offset removal and activation conversion, which grow with
    // the tokens, stay small), else bf16 (no conversion of the activations;
    // measured faster from 4 tokens, and at any M for G = 32).
    // W4_GEMV_F16=0/1 overrides where the group size allows.
    const char* ef = std::getenv("W4_GEMV_F16");
    // K splits added in a cluster where they fit, for 3-8 tokens (measured:
    // 11% faster than the global hand-off on the 12B down projection at 4
    // tokens; 2.6% slower on the 7B step at one token, whose launches
    // overlap the previous kernel's tail, which whole clusters wait out;
    // slower at 16 tokens, where the one-wave limit leaves SMs idle).
    // W4_GEMV_CSPLIT=0 turns it off, =1 allows it at any M.
    const char* ec = std::getenv("W4_GEMV_CSPLIT");
    const bool csplit_ok = act_bytes == 2 && groups == 0 &&
                           (ec ? std::atoi(ec) == 1 : (M >= 3 && M <= 8));
    const bool f16 = act_bytes == 2 && G % 64 == 0 && (ef ? std::atoi(ef) == 1 : M <= 2);
    const int gq = G / 32;
    const int cpg = (gq % 8 == 0) ? 8 : (gq % 4 == 0) ? 4 : (gq % 2 == 0) ? 2 : 1;
    // the fp16 path also keeps four floats per token and segment of cpg*32
    // columns
    auto xseg_bytes = [&](int slice) -> size_t {
        return f16 ? (size_t)M * (slice / (cpg * 32)) * 16 : 0;
    };
    // cross-warp reduction buffer: per thread NT*4 floats (W4A16) or MT*2 ints (W4A8)
    const int red = act_bytes == 2
        ? CW * 32 * ((M > 8 ? 2 : 1) * 4) * 4
        : CW * 32 * (M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16) * 2 * 4;
    // grouped plans keep a list of (group, token tile) items (int32) after the
    // activations; `groups` is its capacity
    const size_t list_bytes = groups > 0 ? (((size_t)groups * 4 + 15) & ~(size_t)15) : 0;
    const size_t fixed = 1024 + (size_t)NS * STAGE_BYTES + kCtlBytes + red + list_bytes;
    const double wbytes = (double)N * Kp / 2.0;
    const double bw_total = 6.5e12, bw_sm = 70e9;
    double best = 1e30;
    bool found = false;
    // two CTAs per SM only for the kernel instances compiled for it
    const int cps_max = (act_bytes == 2 ? M <= 8 : M <= 4) ? 2 : 1;
    // W4_GEMV_ROWS (16, 32, 64 or 128) and W4_GEMV_SPLIT (K splits) pin the
    // plan for tuning sweeps and tests
    auto env_int = [](const char* name) {
        const char* e = std::getenv(name);
        return e ? std::atoi(e) : 0;
    };
    const int fr = env_int("W4_GEMV_ROWS");
    const int forced_r = (fr == 16 || fr == 32 || fr == 64 || fr == 128) ? fr : 0;
    const int forced_s = std::max(env_int("W4_GEMV_SPLIT"), 0);
    const int forced_cps = env_int("W4_GEMV_CPS");      // CTAs of this kernel per SM
    for (int cps = cps_max; cps >= 1; --cps) {
        if ((forced_cps == 1 || forced_cps == 2) && cps != forced_cps) continue;
        // per-CTA shared memory: two CTAs share the SM's 228 KB (1 KB reserved each)
        const size_t cap = cps == 2 ? 115712 : 232448;
        if (fixed >= cap) continue;
        const long per_tok = (long)((cap - fixed) / (size_t)M) - pad;
        for (int R = 16; R <= 128; R *= 2) {
            if (forced_r && R != forced_r) continue;
            const int SKE = 32768 / R;
            const int nst = (Kp + SKE - 1) / SKE;
            const int NB = (N + R - 1) / R;
            const int spl_max =
                (int)(per_tok / ((long)SKE * act_bytes + (f16 ? SKE / (2 * cpg) : 0)));
            if (spl_max < 1) continue;
            const int s_min = (nst + spl_max - 1) / spl_max;
            for (int S = s_min; S <= nst && S <= s_min + 64; ++S) {
                const int spl = (nst + S - 1) / S;
                const int Se = (nst + spl - 1) / spl;
                if (spl > spl_max) continue;
                // the last 34 counters of the prefix belong to the SwiGLU
                // call with INT8 outputs (token maxima, generation, arrival
                // count), never to a row block
                if ((forced_s && Se != forced_s) || (Se > 1 && NB > kMaxCounters - 34) ||
                    (groups > 0 && Se > 1)) {
                    if (Se == nst) break;
                    continue;
                }
                const int units = NB * Se;
                const int grid = std::min(units, cps * sm_count);
                const int per_cta = (units + grid - 1) / grid;
                const int ctas_on_sm = (grid + sm_count - 1) / sm_count;
                const double unit_bytes = (double)R * std::min(spl * SKE, Kp) / 2.0;
                const double sm_bytes = (double)per_cta * ctas_on_sm * unit_bytes;
                // cluster split: up to 8 splits, one wave, the other ranks'
                // sums in rank 0's shared memory (the k-phase register layout)
                const size_t crecv = (size_t)(Se - 1) * (R / 16) * (M > 8 ? 2 : 1) * 512;
                const bool csplit = csplit_ok && !f16 && Se > 1 && Se <= 8 && units <= grid &&
                                    fixed + (size_t)M * (spl * SKE * act_bytes + pad) +
                                            xseg_bytes(spl * SKE) + crecv <= cap;
                double t = std::max(wbytes / bw_total, sm_bytes / bw_sm);
                if (f16) {
                    // one or two tokens: the stream is the whole cost, so
                    // CTAs spread unevenly over the SMs (the busiest SMs set
                    // the pace) and one CTA's own rate (~35 GB/s) count too
                    const double imb = (double)ctas_on_sm * sm_count / grid;
                    t = std::max({wbytes / bw_total * imb, sm_bytes / bw_sm,
                                  per_cta * unit_bytes / 35e9});
                }
                // the hand-off of the splits: a global ticket and a round
                // trip of partial sums, or (cluster) one arrival in
                // distributed shared memory
                t += per_cta * 0.3e-6 + (Se > 1 ? (csplit ? 0.9e-6 : 1.5e-6) : 0.0);
                // the global hand-off reads back every split's partials
                // (measured on the 7B down projection: 64-row blocks split 5
                // ways 11.5 us, 128-row blocks split 10 ways 12.0 us)
                if (Se > 1 && !csplit) t += 0.08e-6 * (Se - 1);
                // every CTA waits for the activation slice of its units (and
                // on the fp16 path converts it: measured ~0.13 ns per column
                // and token)
                if (act_bytes == 2)
                    t += per_cta * (0.3e-6 + (f16 ? 0.13e-9 : 0.02e-9) *
                                                 (double)std::min(spl * SKE, Kp) * M);
                if (t < best * (1 - 1e-9)) {
                    best = t;
                    found = true;
                    GemvPlan p;
                    p.R = R; p.SKE = SKE; p.NB = NB; p.nst = nst; p.S = Se; p.spl = spl;
                    p.units = units; p.grid = grid; p.cps = cps; p.red = red;
                    p.XS = spl * SKE * act_bytes + pad;
                    p.smem = fixed + (size_t)M * p.XS + xseg_bytes(spl * SKE);
                    p.f16 = f16;
                    p.csplit = csplit;
                    if (csplit) {
                        p.smem += crecv;
                        p.crecv_off = p.smem - 1024 - crecv;   // from the aligned base
                    }
                    p.list_off = p.smem - list_bytes - 1024;
                    p.ws_bytes = 0;
                    if (Se > 1) p.ws_bytes = kCounterBytes + (size_t)Se * M * N * 4;
                    *out = p;
                }
                if (Se == nst) break;
            }
        }
    }
    return found;
}
}  // namespace

int launch_w4a16_gemv(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                      cudaStream_t st) {
    if (a.S > 1) return launch_w4a16_gemv_split(packed, a, p, st);
    return launch_w4a16_variant<false>(packed, a, p, st);
}

int launch_w4a8_gemv(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                     cudaStream_t st) {
    if (a.M <= 1) return launch(k_w4a8_gemv_m4<1>, packed, a, p, st);
    if (a.M <= 2) return launch(k_w4a8_gemv_m4<2>, packed, a, p, st);
    if (a.M <= 4) return launch(k_w4a8_gemv_m4<4>, packed, a, p, st);
    if (a.M <= 8) return launch(k_w4a8_gemv_m16<8>, packed, a, p, st);
    return launch(k_w4a8_gemv_m16<16>, packed, a, p, st);
}

}  // namespace w4

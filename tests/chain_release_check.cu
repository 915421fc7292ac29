// Host-only check of the decode chain's release marking (which dependency
// groups publish their completion with a GPU-scope release) against brute
// force over random chains whose buffers overlap.  Built and run by
// test_chain_release_marking.py; makes no CUDA call.
#include "../affine_bit_quantized_gb300/csrc/qmv_chain.cu"

#include <cstdio>
#include <random>

namespace aq {
// the chain source calls the tensor-map encoder only from chain_encode, which this check does not run
bool encode_codes_3d(CUtensorMap *, const void *, uint64_t, uint64_t) { return false; }
}  // namespace aq

using namespace aq;

static bool ov(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

int main() {
    std::mt19937_64 rng(7);
    int bad = 0, released = 0, groups = 0;
    for (int trial = 0; trial < 3000; ++trial) {
        const int n = 1 + (int)(rng() % 40);
        const bool nv = trial % 3 == 0;
        std::vector<aq_matmul_desc> d((size_t)n);
        for (int i = 0; i < n; ++i) {
            aq_matmul_desc &e = d[(size_t)i];
            e.M = 1 + (int64_t)(rng() % 4);
            e.N = 32 * (1 + (int64_t)(rng() % 4));
            e.K = 512 * (1 + (int64_t)(rng() % 2));
            // activations and outputs in one 64 KB arena, so that they overlap often; weights apart,
            // except that now and then an output lands on a weight or the tensor scale
            e.x = reinterpret_cast<const void *>((uintptr_t)(0x100000 + 16 * (rng() % 4096)));
            e.y = reinterpret_cast<void *>((uintptr_t)(0x100000 + 16 * (rng() % 4096)));
            e.w_packed = reinterpret_cast<const uint32_t *>((uintptr_t)(0x10000000 + 0x100000 * (uint64_t)i));
            e.scales = reinterpret_cast<const void *>((uintptr_t)(0x20000000 + 0x100000 * (uint64_t)i));
            e.biases = reinterpret_cast<const void *>((uintptr_t)(0x30000000 + 0x100000 * (uint64_t)i));
            if (rng() % 29 == 0) e.y = const_cast<void *>(reinterpret_cast<const void *>(d[(size_t)(rng() % n)].w_packed));
            if (nv && rng() % 29 == 0) e.y = const_cast<void *>(d[(size_t)(rng() % n)].biases);
            e.flags = (i > 0 && rng() % 3 == 0) ? AQ_CHAIN_INDEPENDENT : 0;
            if (rng() % 17 == 0) e.flags |= AQ_CHAIN_RELEASE;
        }
        std::vector<ChainRec> recs((size_t)n);
        for (ChainRec &r : recs) r.flags = 0;
        std::vector<Span> spans((size_t)n * 5);
        std::vector<int> active((size_t)n * 5), latest((size_t)n), cover((size_t)n + 1);
        mark_releases(d.data(), n, 4, nv, recs.data(), {spans.data(), active.data(), latest.data(), cover.data()});

        // brute force: a group ending at j (not the last) is released iff it is forced or some
        // matmul i <= j and some matmul k > j share memory with at least one of them writing it
        std::vector<Footprint> fp;
        for (int i = 0; i < n; ++i) fp.push_back(footprint(d[(size_t)i], 4, nv));
        auto hazard = [&](int i, int k) {
            const Footprint &a = fp[(size_t)i], &b = fp[(size_t)k];
            if (ov(a.w[0], a.w[1], b.w[0], b.w[1])) return true;
            for (int q = 0; q < 4; ++q)
                if (ov(a.w[0], a.w[1], b.r[q][0], b.r[q][1]) || ov(a.r[q][0], a.r[q][1], b.w[0], b.w[1]))
                    return true;
            return false;
        };
        bool forced = false;
        for (int j = 0; j < n; ++j) {
            forced = forced || (d[(size_t)j].flags & AQ_CHAIN_RELEASE) != 0;
            const bool end = j + 1 == n || !(d[(size_t)j + 1].flags & AQ_CHAIN_INDEPENDENT);
            if (!end) continue;
            bool need = false;
            if (j + 1 < n) {
                need = forced;
                for (int i = 0; i <= j && !need; ++i)
                    for (int k = j + 1; k < n && !need; ++k) need = hazard(i, k);
            }
            const bool got = (recs[(size_t)j].flags & kRecRelease) != 0;
            bad += got != need;
            released += got;
            ++groups;
            forced = false;
        }
    }
    printf("groups %d released %d mismatches %d\n", groups, released, bad);
    return bad != 0 || released == 0 || released == groups;
}

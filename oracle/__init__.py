"""CPU oracle for the wave-index hot path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, double-precision (numpy float64) statement of what the path
computes, written from the RetroInfer summaries (wave index: tripartite
attention approximation, accuracy-bounded estimation, segmented spherical
k-means).  It exists to check the CUDA path; it is not part of the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import or call anything in this package.  It shares no code with the
CUDA path (``clustered_sparse_kv_gb300``) and neither imports the other; the
only common module is the seeded input generator ``kvsynth``.

Parity status per function (what pins it is in ``tests/test_oracle_pins.py``):
  bf16_round          pinned (torch's float32->bfloat16 cast; hand values)
  assign / update     pinned (exhaustive argmax; planted clusters; objective)
  build_unit_index    pinned (conservation invariants; singleton clusters)
  decode_unit         pinned (all-clusters = textbook softmax attention;
                              singleton clusters exact; Jensen bound; cosh
                              closed form; explicit per-token loop); its
                              group-shared top-k variant pinned (one head =
                              the default; brute-force summed-score top-k;
                              all clusters = full attention)
  lse_merge           pinned (associativity against the single sum)
  grow_unit_index     pinned (a grown segment equals build_unit_index of
                              that segment alone; all clusters after growth
                              = textbook softmax; singleton grown clusters
                              make the estimate exact; the window keeps W to
                              W + S - 1 rows)
  full_attention      pinned (equals decode_unit with every cluster
                              retrieved; one row gives its value row;
                              identical keys give the mean value row;
                              row-order invariance)
  LruPagePolicy       pinned in tests/test_oracle_wave_buffer.py (hand-worked
                              LRU trace; a second, stamp-and-argmin statement
                              of the rounds over random traces; cache as
                              large as the working set never evicts, no
                              slots never admits)
Approximation quality against full attention on synthetic data: parity
unpinned (the summaries claim accuracy only on RULER / Needle-in-a-Haystack
with trained models).
tests/test_oracle_mutations.py plants plausible slips in this package's source
and requires each to turn one of those pins red.
"""
from .bf16 import bf16_round, bf16_from_bits, bf16_to_bits, fp32_round  # noqa: F401
from .wave_index import (  # noqa: F401
    IndexParams,
    steady_positions,
    window_start,
    indexed_positions,
    grown_segments,
    grow_unit_index,
    budget_k,
    init_centroids,
    assign,
    update,
    spherical_kmeans,
    build_unit_index,
    build_index,
    select_topk,
    zone_partial,
    lse_merge,
    decode_unit,
    decode,
    full_attention,
)
from .wave_buffer import LruPagePolicy, pages_of_rows  # noqa: F401

"""CPU oracle for the Polestar drift-scoring / sparse-refresh path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``drift_aware_kv_spherical_gb300`` and its CUDA
library) never imports, links or calls it, and this package imports nothing
from the product; the two share no code.  Seeded input generators live in
``drift_aware_kv_spherical_gb300.workloads`` and hold none of the method's
arithmetic.

Source of the method.  Every function cites the page it restates:
"Polestar: Drift-Aware Cache Calibration and Token Commitment for Efficient
Inference of Diffusion LLMs" (gist.science explainer of arXiv 2607.14107),
technical summary, written below as ``[Polestar §x, <paragraph>]``:

* §2.A "Drift measurement"        D_i^(t) = KL(A_i^(t) || A_i^(t-1))
* §2.A "Local window & clustering" spherical k-means, NVFP4 residuals
* §2.A "Sparse updates"           proxy attention on centroids, top-k
                                   drifting clusters, sparse K/V refresh
* §2.B "Current block commitment"  drift delta vs alpha (tau_s - c)^2
* §2.B "Suffix block commitment"   suffix tokens need c >= tau_s
* §2.C "CPU offloading"            quantised clusters in host memory, the
                                   top-k clusters fetched back
* §2.A "schedule"                 refresh after tau_upd decoded tokens,
                                   periodic full passes, window slide
* §2.A / §4 "ablation studies"    cosine-dissimilarity and entropy drift
                                   signals on the proxy distributions

Where the page is silent the oracle takes one explicit reading; each reading
is named in the docstring of the function that takes it.

Precision: fp64 throughout, except the NVFP4 residual, which the format fixes
in fp32 (IEEE round-to-nearest-even for every operation), so that its integer
outputs can be compared bit for bit.

Pins (tests/test_oracle_*.py) tie every function to something other than
itself: closed forms, invariants, brute force and hand-worked fixtures under
``tests/golden/``.  No function here is "parity unpinned".
"""

from .kmeans import kmeans_spherical, kmeanspp_init, normalize_rows
from .nvfp4 import (e2m1_encode, e2m1_decode, e4m3_encode, e4m3_decode,
                    nvfp4_residual, nvfp4_quantize)
from .proxy_kl import centroid_keys, proxy_attn_kl, kl_divergence_rows
from .topk import topk_drift
from .refresh import refresh_kv, bf16_round
from .commit import confidence, commit_rule, CommitParams
from .offload import record_bytes, pack_clusters, reconstruct_row, fetch_reconstruct

__all__ = [
    "kmeans_spherical", "kmeanspp_init", "normalize_rows",
    "e2m1_encode", "e2m1_decode", "e4m3_encode", "e4m3_decode",
    "nvfp4_residual", "nvfp4_quantize",
    "centroid_keys", "proxy_attn_kl", "kl_divergence_rows",
    "topk_drift", "refresh_kv", "bf16_round",
    "confidence", "commit_rule", "CommitParams",
    "record_bytes", "pack_clusters", "reconstruct_row", "fetch_reconstruct",
]
from .schedule import ScheduleState, schedule_step, block_progress
from .scorers import SCORER_KL, SCORER_COSINE, SCORER_ENTROPY, drift_score

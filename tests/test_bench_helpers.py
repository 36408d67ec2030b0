"""Host-side helpers of bench.py (no GPU): kernel names map to the keys the
JSON line reports, the algorithmic work of the dominant kernels matches its
closed form at the LLaDA-8B layer, and the workload config names the logits
dtype and the L2 flush."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from drift_aware_kv_spherical_gb300 import workloads as wl  # noqa: E402


def test_kernel_names_map_to_report_keys():
    cases = {
        "void ps::k_tc_gemm<256, 1, 1, 1, ps::RefreshClusterEpi<256>>(...)": "refresh_gemm",
        "ps::<unnamed>::k_km_gram(...)": "kmeans_passes",
        "void ps::k_tc_gemm<128, 1, 1, 0, ps::GramClusterEpi>(...)": "gram_gemm",
        "_ZN2ps47_GLOBAL__N__329e6c79_14_kmeans_gram_cu_4b96a88010k_kpp_gramEPK13__nv_bfloat16":
            "kpp_gram",
        "ps::<unnamed>::k_drift_score(const float *, ...)": "drift_score",
        "void ps::<unnamed>::k_commit_scan<__nv_bfloat16, 8>(...)": "commit_scan",
        "void ps::<unnamed>::k_pack_clusters(...)": "offload_pack",
        "void ps::<unnamed>::k_fetch_dequant(...)": "offload_fetch",
        "_ZN2ps12_GLOBAL__N_114k_cluster_scanI13__nv_bfloat16Lb0ELb1ELb1EEEvv": "kmeans_update",
        "_ZN2ps12_GLOBAL__N_114k_cluster_scanI13__nv_bfloat16Lb1ELb0ELb0EEEvv": "kmeans_final",
        "ps::<unnamed>::k_km_fin_stats(const int *, ...)": "kmeans_fin_stats",
        "ps::<unnamed>::k_km_fin_chat(const int *, ...)": "kmeans_final",
        "ps::<unnamed>::k_km_rho(const __nv_bfloat16 *, ...)": "kmeans_rho",
        "ps::<unnamed>::k_gather_rows(const __nv_bfloat16 *, ...)": "refresh_gather",
    }
    for name, key in cases.items():
        assert bench.kernel_key(name) == key, name


def test_refresh_and_commit_work_closed_forms():
    w = wl.BY_NAME["llada8b_layer_n1024"]
    M = 147.0
    by, fl = bench.kernel_work("refresh_gemm", w, M)
    nkv = w.Hkv * w.dh
    assert by == 2 * w.d * nkv * 2 + M * w.d * 2 + 2 * M * nkv * 2
    assert fl == 4.0 * M * w.d * nkv
    assert bench.kernel_work("commit_scan", w, M)[0] == w.B * w.P * w.V * 2   # bf16 logits
    tiny = wl.BY_NAME["tiny_d256_n128"]
    assert bench.kernel_work("commit_scan", tiny, 1)[0] == tiny.B * tiny.P * tiny.V * 4
    # bf16 windows with fp32 logits: the scan's bytes are the logits' own
    st = wl.BY_NAME["stress_b32_n4096_l32"]
    assert st.dtype == "bf16" and st.logits == "f32"
    assert bench.kernel_work("commit_scan", st, 1)[0] == st.B * st.P * st.V * 4
    assert bench.op_work(st, 1)["commit"][0] == st.B * st.P * st.V * 4
    assert bench.kernel_work("no_such_kernel", w, M) is None


def test_workload_config_names_logits_and_flush():
    cfg = bench.workload_config(wl.BY_NAME["llada8b_layer_n1024"])
    assert cfg["workload"] == "llada8b_layer_n1024" and cfg["logits"] == "bf16"
    assert "flushed" in cfg["l2"]
    assert bench.L2_FLUSH_BYTES > 129 * 10**6      # larger than the GPU's L2

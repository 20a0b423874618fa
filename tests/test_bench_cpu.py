"""CPU tier of bench.py's roofline arithmetic: the algorithmic bytes and flops
of the layer against figures worked out by hand from the layer's definition
(per routed expert: gate_up 2·I·d and down d·I weights; int4 as two codes per
byte plus one bf16 scale per 32 codes), and the traffic record's source check."""
import json

import numpy as np
import pytest

import bench
from moe_expert_layer_gemv_gb300 import inputs as I

MiB = 1 << 20


def ids_with(n_experts, T, k):
    """Routing that touches experts 0..n_experts-1 (each token's k distinct)."""
    return np.array([[(t * k + j) % n_experts for j in range(k)] for t in range(T)], np.int32)


def test_verify_t8_bytes_by_hand():
    s = I.shape("verify_t8")
    ids = ids_with(57, s.T, s.k)
    a = bench.algorithmic(s, [ids])
    # one bf16 routed expert: gate_up 4 MiB + down 2 MiB = 6,291,456 B
    per_expert = 6 * MiB
    shared = 4 * MiB + 2 * MiB + 2048 * 2          # shared gate_up, down, w_sg
    router = 256 * 2048 * 2                         # 1 MiB
    x = out = 8 * 2048 * 2
    assert a["touched"] == 57
    assert a["layer_bytes"] == 57 * per_expert + shared + router + x + out
    assert a["gate_up_bytes"] == 57 * 4 * MiB + 4 * MiB + x
    # 2·slots·3·I·d + 2·T·3·I_s·d + 2·T·E·d
    assert a["flops"] == 2 * 64 * 3 * 512 * 2048 + 2 * 8 * 3 * 512 * 2048 + 2 * 8 * 256 * 2048


def test_int4_t32_bytes_by_hand():
    s = I.shape("int4_t32")
    ids = ids_with(237, s.T, s.k)
    a = bench.algorithmic(s, [ids])
    # one int4 routed expert: codes 2·512·2048/2 + 2048·512/2 = 1,572,864 B,
    # scales (2·512·64 + 2048·16)·2 = 196,608 B -> 1,769,472 B
    per_expert = 1_769_472
    shared = 2 * 1024 * 2048 * 2 + 2048 * 1024 * 2 + 2048 * 2   # 12 MiB + w_sg
    router = 512 * 2048 * 2
    x = out = 32 * 2048 * 2
    assert a["layer_bytes"] == 237 * per_expert + shared + router + x + out
    assert a["gate_up_bytes"] == 237 * (1_048_576 + 131_072) + 2 * 1024 * 2048 * 2 + x


def test_touched_experts_average_over_batches():
    s = I.shape("verify_t8")
    a = bench.algorithmic(s, [ids_with(10, s.T, s.k), ids_with(20, s.T, s.k)])
    assert a["touched"] == 15
    assert a["layer_bytes"] == (bench.algorithmic(s, [ids_with(10, s.T, s.k)])["layer_bytes"] +
                                bench.algorithmic(s, [ids_with(20, s.T, s.k)])["layer_bytes"]) / 2


def test_prefill_gate_up_flops_and_dispatch():
    s = I.shape("prefill_t4096")
    assert bench.gate_up_flops(s) == 2 * 4096 * 8 * 1024 * 2048 + 2 * 4096 * 1024 * 2048
    assert bench.tensor_core_path(s)
    assert not bench.tensor_core_path(I.shape("verify_t8"))
    assert not bench.tensor_core_path(I.shape("int4_t32"))


def test_traffic_record_scales_and_checks_source(tmp_path, monkeypatch):
    src_dir = tmp_path / "moe_expert_layer_gemv_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (src_dir / "k.cu").write_text("kernel v1\n")
    import hashlib
    h = hashlib.sha256(b"kernel v1\n").hexdigest()
    rec = {"dram_bytes_per_launch": 1100, "algorithmic_bytes_of_capture": 1000,
           "source_sha256": h}
    (tmp_path / "profiles" / "gate_up_w.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("k.cu", "w", 2000) == pytest.approx(2200)
    (src_dir / "k.cu").write_text("kernel v2\n")  # source changed since the capture
    assert bench.kernel_traffic("k.cu", "w", 2000) is None
    assert bench.kernel_traffic("k.cu", "missing", 2000) is None

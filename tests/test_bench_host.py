"""Host-side arithmetic of bench.py, on the CPU: the algorithmic bytes and MMA
flops the roofline divides by, and the code hash that keys recorded traffic."""
import os
import shutil

import numpy as np

import bench
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bytes_per_cached_token():
    # a cached token is its latent + RoPE row in the cache dtype plus G fp32 alpha^k
    w = W.WORKLOADS[2]                                    # d_c 512, d_r 64, G 8, bf16
    lens = np.array([1000])
    b, _, kv = bench.algorithmic(w.with_(B=1), lens)
    assert kv == 1000 * ((512 + 64) * 2 + 8 * 4)          # 1184 B a token
    _, _, kv_plain = bench.algorithmic(w.with_(B=1), lens, plain=True)
    assert kv_plain == 1000 * (512 + 64) * 2              # plain MLA reads no alpha
    w1 = W.WORKLOADS[1]                                   # d_c 256, d_r 32, G 4, bf16
    _, _, kv1 = bench.algorithmic(w1.with_(B=1), lens)
    assert kv1 == 1000 * ((256 + 32) * 2 + 4 * 4)         # 592 B a token


def test_decode_call_bytes_and_flops_of_the_dsv3_batch():
    # 64 sequences of 4096 tokens, 128 heads: cache once, queries and outputs once
    w = W.WORKLOADS[2]
    lens = W.seq_lens(w)
    assert int(lens.sum()) == 64 * 4096
    b, f, kv = bench.algorithmic(w, lens)
    rows = 64 * 128
    q_side = rows * (512 * 2 + 4 + 64 * 4)                # q~ bf16, alpha^q, q_rope fp32
    out = rows * (512 * 4 + 4)                            # o fp32 + lse
    assert kv == 64 * 4096 * 1184
    assert b == kv + q_side + out == 337_707_008
    # logit (content + RoPE) and output MMAs per visible (token, head)
    assert f == 64 * 4096 * 128 * 2 * (2 * 512 + 64) == 73_014_444_032


def test_causal_visibility_with_two_query_tokens():
    # query i of a sequence of length L sees L - s_q + i + 1 tokens
    w = W.WORKLOADS[4].with_(B=2)
    lens = np.array([10, 100])
    _, f, _ = bench.algorithmic(w, lens)
    visible = (9 + 10) + (99 + 100)
    assert f == visible * w.H * 2 * (2 * w.d_c + w.d_r)


def test_code_hash_ignores_comments_and_layout(tmp_path):
    src = os.path.join(bench.ROOT, "qk_normed_latent_gb300", "csrc")
    dst = tmp_path / "csrc"
    shutil.copytree(src, dst)
    base = bench.kernel_signature(str(dst))
    assert base == bench.kernel_signature()
    f = dst / "decode_tc.cu"
    text = f.read_text()
    f.write_text("// a new leading comment\n/* and a block\n   comment */\n" + text.replace(";\n", ";\n\n", 3))
    assert bench.kernel_signature(str(dst)) == base        # comments and blank lines only
    f.write_text(text.replace("constexpr int kThreads = 192;", "constexpr int kThreads = 256;"))
    assert bench.kernel_signature(str(dst)) != base        # a code change


def test_cpu_baseline_always_times_at_least_one_sequence():
    # the reference arm's warm-up asks for a zero-second sample
    w = W.small(W.WORKLOADS[0], 1, (64,))
    rate, sample, secs, busy = bench.cpu_oracle_rate(w, 0.0)
    assert rate > 0 and secs > 0
    assert sample.startswith("1 sequence steps")
    assert busy > 0


def test_reference_arm_reports_the_same_config():
    """Both arms print the same `config` object for a workload, so the driver can
    pair them."""
    import json
    import subprocess
    import sys
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "0",
                          "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.05"],
                         capture_output=True, text=True, check=True).stdout
    line = json.loads(out.strip().splitlines()[-1])
    w = W.WORKLOADS[0]
    assert line["impl"] == "reference"
    assert line["config"] == bench.config_of(w, W.seq_lens(w), 1)
    assert line["cpu_baseline"]["cores"] >= 1

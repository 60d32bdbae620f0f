"""Host-side logic of bench.py that needs no GPU."""

import bench


def test_source_digest_ignores_comments_and_whitespace_only():
    """A traffic figure stays attached to the kernels' code: editing comments
    or whitespace keeps the digest's input, changing code does not."""
    base = 'int f(int a) {  // add one\n  return a + 1; /* done */\n}\nconst char* s = "x//y";\n'
    comments = '/* header */\nint f(int a) {\n  // add one to a\n      return a + 1;\n}\n\nconst char* s = "x//y";\n'
    code = 'int f(int a) {  // add one\n  return a + 2; /* done */\n}\nconst char* s = "x//y";\n'
    literal = 'int f(int a) {  // add one\n  return a + 1; /* done */\n}\nconst char* s = "x/y";\n'
    assert bench._code_only(base) == bench._code_only(comments)
    assert bench._code_only(base) != bench._code_only(code)
    assert bench._code_only(base) != bench._code_only(literal)
    assert bench._code_only("char c = '\\'';  // quote\nint x;") == "char c = '\\'';\nint x;"



def test_source_digest_per_kernel_family():
    """A traffic row is keyed on its kernel family's sources: the digest of
    one family covers its own files and the shared ones, and differs between
    families and from the whole library's."""
    fams = {f: bench.library_source_hash(f) for f in bench.KERNEL_SOURCES}
    assert len(set(fams.values())) == len(fams)
    assert bench.library_source_hash() not in fams.values()
    assert bench.library_source_hash("chunked") == bench.library_source_hash("chunked")


def test_decode_and_verify_bytes_are_the_component_sums():
    """KDA decode at Kimi-K3 TP8 shard shapes (12 heads x 128, bf16, per-key
    gates): per request-step the state read and written (2 x 393,216), the
    conv window read and written (2 x 27,648), x 9,216, g 6,144, beta 48, the
    output 3,072 and the track copy amortised over 256 steps (420,864 / 256);
    a verify of 4 drafts reads the state and window once and writes four."""
    import workloads as W
    dims = W.KIMI_K3_TP8
    step, launch = bench.decode_algo_bytes(dims, 256, 1)
    per = 2 * 393216 + 2 * 27648 + 9216 + 6144 + 48 + 3072 + 420864 / 256
    assert per == 861852
    assert step == launch == 256 * per
    total, verify = bench.decode_algo_bytes(dims, 256, 4)
    assert verify == 256 * ((393216 + 27648) * (1 + 4) + 4 * (9216 + 6144 + 48) + 4 * 3072)
    assert verify / 256 == 2178240
    assert total == verify + 256 * 2 * (393216 + 27648)
    _, tree8 = bench.decode_algo_bytes(dims, 256, 8)
    assert tree8 == 256 * ((393216 + 27648) * 9 + 8 * (9216 + 6144 + 48 + 3072))
    _, replay = bench.decode_algo_bytes(dims, 256, 4, replay=True)
    assert replay == 256 * ((393216 + 27648) + 4 * (9216 + 6144 + 48 + 3072))


def test_prefill_bytes_are_the_component_sums():
    """Qwen3.5-style GDN prefill (32 heads x 128, bf16 x, fp32 state and
    outputs, 8 x 4096 tokens, cold, snapshot every 64): per token x 24,576,
    g 128, beta 128, output 16,384; 512 snapshots and 8 final write-backs of
    one state block (2,097,152 + 73,728); the conv taps 12,288 x 4 x 2."""
    import workloads as W
    b, n_snap = bench.prefill_algo_bytes(W.QWEN35_GDN, [4096] * 8, [0] * 8, [0] * 8,
                                         W.GATE_PER_HEAD, 2, 4, 4, 64)
    assert n_snap == 512
    assert b == (32768 * (24576 + 128 + 128 + 16384) + (512 + 8) * (2097152 + 73728)
                 + 12288 * 4 * 2)
    # a warm request adds its initial state read; a 64-multiple prefix moves
    # the boundaries with it
    b2, n2 = bench.prefill_algo_bytes(W.QWEN35_GDN, [4096], [64], [1], W.GATE_PER_HEAD,
                                      2, 4, 4, 64)
    assert n2 == 64
    assert b2 == 4096 * (24576 + 128 + 128 + 16384) + (64 + 1 + 1) * (2097152 + 73728) + 12288 * 8

"""Host-side path policy of binding.ffn_forward(path="auto") (no GPU)."""
from activation_sparse_ffn_gate_gb300 import binding


def test_small_batches_take_the_decode_path():
    for n in (1, 8, binding.DECODE_MAX_N):
        assert binding.choose_path(n, None) == "decode"
        assert binding.choose_path(n, 0.05) == "decode"


def test_density_chooses_walk_or_union():
    n = binding.SMALL_BATCH_MAX_N + 1
    assert binding.choose_path(n, None) == "walk"  # no estimate yet: the walk
    assert binding.choose_path(8192, 0.004) == "walk"
    assert binding.choose_path(8192, 0.005) == "union"
    assert binding.choose_path(8192, 0.01) == "union"
    assert binding.choose_path(n, binding.UNION_MIN_DENSITY) == "union"
    assert binding.choose_path(8192, 0.02) == "union"
    assert binding.choose_path(8192, 0.5) == "union"


def test_batches_up_to_128_tokens_take_the_union_path_at_any_density():
    for n in (binding.DECODE_MAX_N + 1, 64, binding.UNION_ANY_DENSITY_MAX_N):
        for d in (None, 0.0, 0.001, 0.005, 0.5):
            assert binding.choose_path(n, d) == "union"


def test_batches_of_129_to_512_tokens_switch_lower_still():
    assert binding.choose_path(129, None) == "walk"
    assert binding.choose_path(200, 0.0005) == "walk" and binding.choose_path(200, 0.001) == "union"
    assert binding.choose_path(256, 0.0025) == "union"
    assert binding.choose_path(512, 0.001) == "walk" and binding.choose_path(512, 0.0025) == "union"
    assert binding.choose_path(513, 0.0025) == "walk"


def test_batches_up_to_4096_tokens_switch_at_a_lower_density():
    for n in (513, 1024, binding.SMALL_BATCH_MAX_N):
        assert binding.choose_path(n, None) == "walk"
        assert binding.choose_path(n, 0.001) == "walk"
        assert binding.choose_path(n, 0.005) == "union"
        assert binding.choose_path(n, binding.UNION_MIN_DENSITY_SMALL_BATCH) == "union"

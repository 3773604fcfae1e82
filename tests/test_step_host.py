"""Host logic of the captured-step set: size choice and cohort splitting."""
from decode_step_gb300.step import choose_size, cohorts


def test_choose_size():
    sizes = [1, 4, 16, 64]
    assert [choose_size(sizes, n) for n in (1, 2, 4, 5, 16, 17, 64, 65)] == [1, 4, 4, 16, 16, 64, 64, None]


def test_cohorts_cover_every_stream_once():
    for n in (0, 1, 63, 64, 65, 128, 200):
        parts = cohorts(n, 64)
        assert sum(c for _, c in parts) == n
        assert all(0 < c <= 64 for _, c in parts)
        assert [f for f, _ in parts] == list(range(0, n, 64))

"""The float64 oracle of the fused prologue against its pins (CPU only)."""
import _pins_prologue as pp


def test_norm_at_position_zero_is_torch_rms_norm():
    pp.check_norm_at_position_zero()


def test_rotation_keeps_pair_norms():
    pp.check_rotation_keeps_pair_norms()


def test_scores_depend_on_relative_position_only():
    pp.check_relative_position()

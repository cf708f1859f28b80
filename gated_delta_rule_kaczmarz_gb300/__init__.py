"""Kaczmarz Linear Attention for GB300 (sm_103a)."""

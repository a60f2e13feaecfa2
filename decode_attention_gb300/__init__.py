"""GB300 (sm_103a) decode-step attention core for the Gemma-4-31B text decoder."""
